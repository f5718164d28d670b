"""Grouped FP8 MoE path on the GPU vs the FP64 oracle ("DeepGEMM teardown
(FP8 GEMM)", sections 2.2 and 5.3; "DeepGEMM for Hopper MoE", section 2.1).

The row gather is byte work: bit-exact.  The grouped GEMM is checked per
expert against the oracle's FP8 GEMM on the same codes and scales within
|y - y_ref| <= 1e-3 S + 2^-8 |y_ref| (bf16 output) and the tighter 1e-4 S
diagnostic.  The layer is checked in the same stages as the FP4 layer: routed
activation codes bit-exact, h against the oracle's SwiGLU of its GEMMs on the
GPU's codes, re-quantized h bit-exact against the oracle re-quantizing the
GPU's h, and the combined output against the oracle's down GEMMs on the GPU's
quantized h.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.helpers import gemm_errors, routing, tight_errors

pytestmark = pytest.mark.gpu

ROUTER_RTOL = 4e-6   # as in the FP4 MoE test: fp32 softmax of the chosen logits


def _groups(counts):
    """counts -> (offsets [E+1] with 128-aligned starts, total rows)."""
    offs = [0]
    for c in counts:
        offs.append(offs[-1] + (c + 127) // 128 * 128)
    return np.array(offs, dtype=np.int32)


def _h_bound(g, u, s_g, s_u, h_ref):
    """Error of bf16(silu(g) u) from |g - g_ref| <= 1e-3 S_g and |u - u_ref| <=
    1e-3 S_u (first-order), plus the bf16 rounding of h."""
    sig = 1.0 / (1.0 + np.exp(-g))
    dsilu = np.abs(sig * (1 + g * (1 - sig)))
    return 1e-3 * (dsilu * np.abs(u) * s_g + np.abs(g * sig) * s_u) + 2.0 ** -8 * np.abs(h_ref) + 1e-30


@pytest.mark.parametrize("rows_in,rows_out,K", [(1, 1, 128), (300, 700, 384), (64, 1000, 7168)])
def test_fp8_gather_rows_bit_exact(cuda_lib, rows_in, rows_out, K):
    """Gathered codes and scales equal the oracle quantizing the gathered rows;
    -1 and out-of-range indices give zero rows with zero scales."""
    bs = cuda_lib
    g = torch.Generator().manual_seed(rows_in + rows_out + K)
    x = torch.randn(rows_in, K, generator=g).to(torch.bfloat16)
    idx = torch.randint(-1, rows_in + 2, (rows_out,), generator=g, dtype=torch.int32)
    codes, scales = bs.q8_quantize(x.cuda(), mode=bs.Q8_TOKEN)
    oc, os_ = bs.fp8_gather_rows(codes, scales, idx.cuda())
    torch.cuda.synchronize()
    idx = idx.numpy()
    valid = (idx >= 0) & (idx < rows_in)
    rc, rs = oracle.q8_quantize(x[idx[valid]], 1)
    gc, gs = oc.cpu().numpy(), os_.cpu().numpy().T   # scales back to [rows, K/128]
    assert np.array_equal(gc[valid], rc) and np.array_equal(gs[valid], rs)
    assert np.all(gc[~valid] == 0) and np.all(gs[~valid] == 0)


def _grouped_case(counts, N, K, wrows_per_expert, seed):
    g = torch.Generator().manual_seed(seed)
    E = len(counts)
    offs = _groups(counts)
    M = int(offs[-1]) + 128    # rows past the last segment stay unused
    x = torch.randn(M, K, generator=g)
    x[:, 7] *= 30
    w = torch.randn(E * wrows_per_expert, K, generator=g) * 0.05
    return offs, M, x.to(torch.bfloat16), w.to(torch.bfloat16)


def _quant(bs, x, w):
    xq, xs = bs.q8_quantize(x.cuda(), mode=bs.Q8_TOKEN)
    wq, ws = bs.q8_quantize(w.cuda(), mode=bs.Q8_BLOCK)
    return xq, xs, wq, ws


COUNTS = [[0, 1, 128, 129, 300], [700], [5, 0, 0, 256, 64, 383, 1]]


@pytest.mark.parametrize("counts", COUNTS, ids=["mixed", "one", "sparse"])
@pytest.mark.parametrize("N,K", [(128, 128), (384, 640), (256, 2176)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_grouped_gemm_fp8_store(cuda_lib, counts, N, K, out_dtype):
    """K = 2176: 17 K blocks, more than one 16-block scale chunk plus a tail."""
    bs = cuda_lib
    E = len(counts)
    offs, M, x, w = _grouped_case(counts, N, K, N, sum(counts) + N + K)
    xq, xs, wq, ws = _quant(bs, x, w)
    cnt = torch.tensor(counts, dtype=torch.int32)
    out = torch.full((M, N), 7.0, dtype=out_dtype, device="cuda")
    bs.grouped_gemm_fp8(xq, xs, wq, ws, N=N, E=E, offsets=torch.from_numpy(offs).cuda(), counts=cnt.cuda(),
                        epilogue=bs.EPI_STORE, out=out)
    torch.cuda.synchronize()
    assert bs.device_status()[0] == 0
    a, sa = xq.cpu().numpy(), xs.cpu().numpy().T
    b, sb = wq.cpu().numpy(), ws.cpu().numpy()
    o = out.float().cpu().numpy()
    covered = np.zeros(M, dtype=bool)
    bf = out_dtype == torch.bfloat16
    for e in range(E):
        seg = np.arange(offs[e], offs[e] + counts[e])
        covered[seg] = True
        if len(seg) == 0:
            continue
        yr, s = oracle.gemm_fp8(a[seg], sa[seg], b[e * N:(e + 1) * N], sb[e * N // 128:(e + 1) * N // 128])
        ok, ratio, rel = gemm_errors(o[seg], yr, s, bf)
        tok, tratio = tight_errors(o[seg], yr, s, bf)
        assert ok and tok, (e, ratio, rel, tratio)
    assert np.all(o[~covered] == 7.0)   # rows outside the segments are untouched


@pytest.mark.parametrize("num_sms", [0, 3])
@pytest.mark.parametrize("counts", COUNTS[::2], ids=["mixed", "sparse"])
def test_grouped_gemm_fp8_swiglu(cuda_lib, counts, num_sms):
    """SWIGLU: h = bf16(silu(g) u) with g = rows [0, F) and u = rows [F, 2F)
    of each expert's weights; padding rows of a segment are written as 0.
    num_sms = 3: several tiles per CTA, the scale staging crossing tiles."""
    bs = cuda_lib
    E, F, K = len(counts), 256, 384
    offs, M, x, w = _grouped_case(counts, F, K, 2 * F, 11 + sum(counts))
    xq, xs, wq, ws = _quant(bs, x, w)
    h = torch.full((M, F), 3.0, dtype=torch.bfloat16, device="cuda")
    bs.grouped_gemm_fp8(xq, xs, wq, ws, N=F, E=E, offsets=torch.from_numpy(offs).cuda(),
                        counts=torch.tensor(counts, dtype=torch.int32).cuda(), epilogue=bs.EPI_SWIGLU, out=h,
                        num_sms=num_sms)
    torch.cuda.synchronize()
    assert bs.device_status()[0] == 0
    a, sa = xq.cpu().numpy(), xs.cpu().numpy().T
    b, sb = wq.cpu().numpy(), ws.cpu().numpy()
    hg = h.float().cpu().numpy()
    seg_rows = np.zeros(M, dtype=bool)
    for e in range(E):
        seg = np.arange(offs[e], offs[e] + counts[e])
        blk_end = offs[e] + (counts[e] + 127) // 128 * 128
        seg_rows[offs[e]:blk_end] = True
        assert np.all(hg[offs[e] + counts[e]:blk_end] == 0)   # padding rows of the segment
        if len(seg) == 0:
            continue
        gu, s = oracle.gemm_fp8(a[seg], sa[seg], b[e * 2 * F:(e + 1) * 2 * F],
                                sb[e * 2 * F // 128:(e + 1) * 2 * F // 128])
        g_, u_ = gu[:, :F], gu[:, F:]
        h_ref = oracle.swiglu(g_, u_)
        assert np.all(np.abs(hg[seg] - h_ref) <= _h_bound(g_, u_, s[:, :F], s[:, F:], h_ref)), e
    assert np.all(hg[~seg_rows] == 3.0)


def test_grouped_gemm_fp8_rows(cuda_lib):
    """ROWS: out fp32 [r, n] = weight_of[r] * y[r, n] on the segment rows."""
    bs = cuda_lib
    counts = [200, 0, 77, 129]
    E, N, K = len(counts), 256, 512
    offs, M, x, w = _grouped_case(counts, N, K, N, 99)
    xq, xs, wq, ws = _quant(bs, x, w)
    wt = torch.rand(M, generator=torch.Generator().manual_seed(5)) + 0.25
    out = torch.full((M, N), -1.0, dtype=torch.float32, device="cuda")
    bs.grouped_gemm_fp8(xq, xs, wq, ws, N=N, E=E, offsets=torch.from_numpy(offs).cuda(),
                        counts=torch.tensor(counts, dtype=torch.int32).cuda(), epilogue=bs.EPI_ROWS, out=out,
                        weight_of=wt.cuda())
    torch.cuda.synchronize()
    assert bs.device_status()[0] == 0
    a, sa = xq.cpu().numpy(), xs.cpu().numpy().T
    b, sb = wq.cpu().numpy(), ws.cpu().numpy()
    o = out.cpu().numpy()
    wn = wt.numpy().astype(np.float64)
    for e in range(E):
        seg = np.arange(offs[e], offs[e] + counts[e])
        if len(seg) == 0:
            continue
        yr, s = oracle.gemm_fp8(a[seg], sa[seg], b[e * N:(e + 1) * N], sb[e * N // 128:(e + 1) * N // 128])
        ok, ratio, rel = gemm_errors(o[seg], wn[seg, None] * yr, wn[seg, None] * s, False)
        assert ok, (e, ratio, rel)
        assert np.all(o[offs[e] + counts[e]:offs[e + 1]] == -1.0)


def test_grouped_gemm_fp8_bad_offsets(cuda_lib):
    """An offset that is not a multiple of 128 sets BS_ERR_OFFSETS in the
    device status and the kernel writes nothing."""
    bs = cuda_lib
    counts = [10, 10]
    offs, M, x, w = _grouped_case(counts, 128, 128, 128, 1)
    offs = offs.copy()
    offs[1] = 64
    xq, xs, wq, ws = _quant(bs, x, w)
    out = torch.full((M, 128), 5.0, dtype=torch.bfloat16, device="cuda")
    bs.clear_device_status()
    bs.grouped_gemm_fp8(xq, xs, wq, ws, N=128, E=2, offsets=torch.from_numpy(offs).cuda(),
                        counts=torch.tensor(counts, dtype=torch.int32).cuda(), epilogue=bs.EPI_STORE, out=out)
    torch.cuda.synchronize()
    assert bs.device_status()[0] == bs.BS_ERR_OFFSETS
    bs.clear_device_status()
    assert torch.all(out == 5.0)


def test_grouped_gemm_fp8_rejects(cuda_lib):
    bs = cuda_lib
    offs, M, x, w = _grouped_case([10], 128, 128, 128, 2)
    xq, xs, wq, ws = _quant(bs, x, w)
    o32 = torch.zeros((M, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(bs.BSError) as e:   # COMBINE is FP4 only
        bs.grouped_gemm_fp8(xq, xs, wq, ws, N=128, E=1, offsets=torch.from_numpy(offs).cuda(),
                            counts=torch.tensor([10], dtype=torch.int32).cuda(), epilogue=bs.EPI_COMBINE, out=o32)
    assert e.value.status == bs.BS_ERR_UNSUPPORTED


def _fp8_weights(ws):
    from fp8_quantized_gemm_q4_gb300.moe import quantize_expert_weights_fp8
    return quantize_expert_weights_fp8([a for a, _ in ws], [b for _, b in ws])


def _check_layer_stages(bs, layer, x, ids, wts, ws_host, samples, F, H):
    """Stages on the tokens `samples` (see the module docstring).  ws_host[e] =
    (bf16 gate/up [2F, H], bf16 down [H, F]) of every expert the samples use."""
    k = ids.shape[1]
    rop = layer.row_of_pair.cpu().numpy()
    rows = np.array([rop[t * k + j] for t in samples for j in range(k)])
    assert np.all(rows >= 0)
    ridx = torch.from_numpy(rows).cuda().long()
    xq = layer.xq[ridx].cpu().numpy()
    xs = layer.xs[:, ridx].cpu().numpy().T
    oa, osa = oracle.q8_quantize(x[[t for t in samples for _ in range(k)]], 1)
    assert np.array_equal(xq, oa) and np.array_equal(xs, osa)
    h = layer.h[ridx].float().cpu().numpy()
    hq = layer.hq[ridx].cpu().numpy()
    hs = layer.hs[:, ridx].cpu().numpy().T
    ohq, ohs = oracle.q8_quantize(layer.h[ridx].cpu(), 1)
    assert np.array_equal(hq, ohq) and np.array_equal(hs, ohs)
    experts = sorted({int(e) for t in samples for e in ids[t]})
    oq = {e: (oracle.q8_quantize(ws_host[e][0], 128), oracle.q8_quantize(ws_host[e][1], 128)) for e in experts}
    got = layer.out.float().cpu().numpy()
    for i, t in enumerate(samples):
        ref = np.zeros(H)
        S = np.zeros(H)
        for j in range(k):
            n = i * k + j
            e = int(ids[t, j])
            (gu_c, gu_s), (d_c, d_s) = oq[e]
            gu, s_gu = oracle.gemm_fp8(xq[n:n + 1], xs[n:n + 1], gu_c, gu_s)
            g_, u_ = gu[:, :F], gu[:, F:]
            h_ref = oracle.swiglu(g_, u_)
            assert np.all(np.abs(h[n:n + 1] - h_ref) <= _h_bound(g_, u_, s_gu[:, :F], s_gu[:, F:], h_ref)), (t, j)
            y, sy = oracle.gemm_fp8(hq[n:n + 1], hs[n:n + 1], d_c, d_s)
            wgt = float(wts[t, j])
            ref += wgt * y[0]
            S += abs(wgt) * sy[0]
        ok, ratio, rel = gemm_errors(got[t:t + 1], ref[None], S[None], True)
        assert ok, (t, ratio, rel)


@pytest.mark.parametrize("T,H,F,E,k", [(200, 256, 128, 5, 2), (1000, 512, 256, 8, 4), (64, 384, 128, 16, 8)])
def test_fp8_layer_staged(cuda_lib, T, H, F, E, k):
    bs = cuda_lib
    from fp8_quantized_gemm_q4_gb300.moe import Fp8MoELayer
    r = routing(T, E, k, index=5)
    x = workloads.moe_activations(T, H, index=5)
    ws = [workloads.moe_expert_weights(e, F, H, index=5) for e in range(E)]
    layer = Fp8MoELayer(_fp8_weights(ws), T, k)
    out = layer.forward(x.cuda(), torch.from_numpy(r["topk_ids"]).cuda(), torch.from_numpy(r["topk_w"]).cuda())
    torch.cuda.synchronize()
    assert bs.device_status()[0] == 0
    _check_layer_stages(bs, layer, x, r["topk_ids"], r["topk_w"], ws, list(range(T)), F, H)
    # a second call gives the same output bit for bit
    first = out.clone()
    out2 = layer.forward(x.cuda(), torch.from_numpy(r["topk_ids"]).cuda(), torch.from_numpy(r["topk_w"]).cuda())
    torch.cuda.synchronize()
    assert torch.equal(out2.view(torch.int16), first.view(torch.int16))


def test_fp8_layer_end_to_end_report(cuda_lib):
    """End to end against the oracle's own FP8 layer (its own h and
    re-quantization): looser, reported."""
    bs = cuda_lib
    from fp8_quantized_gemm_q4_gb300.moe import Fp8MoELayer
    T, H, F, E, k = 64, 256, 128, 4, 2
    r = routing(T, E, k, index=6)
    x = workloads.moe_activations(T, H, index=6)
    ws = [workloads.moe_expert_weights(e, F, H, index=6) for e in range(E)]
    out = Fp8MoELayer(_fp8_weights(ws), T, k).forward(x.cuda(), torch.from_numpy(r["topk_ids"]).cuda(),
                                                      torch.from_numpy(r["topk_w"]).cuda())
    torch.cuda.synchronize()
    gu = [oracle.q8_quantize(a, 128) for a, _ in ws]
    dn = [oracle.q8_quantize(b, 128) for _, b in ws]
    ref = oracle.moe_layer(x, r["topk_ids"], r["topk_w"], [c for c, _ in gu], [s for _, s in gu],
                           [c for c, _ in dn], [s for _, s in dn], F=F, fmt="fp8")["out"]
    o = out.float().cpu().numpy()
    rel = np.abs(o - ref).max() / np.abs(ref).max()
    print(f"end-to-end FP8 MoE max |err| / max |ref| = {rel:.3g}")
    assert rel < 0.02
    assert bs.device_status()[0] == 0


def test_fp8_layer_full_size_sampled_tokens(cuda_lib):
    """The 4096-token MoE configuration (H 4096, E 64, k 8, F 1536) in FP8,
    from the router's logits, through the captured CUDA graph the bench
    replays, checked in stages on sampled tokens: first, middle, last, one
    routed to the most loaded expert and one to the least loaded."""
    bs = cuda_lib
    from fp8_quantized_gemm_q4_gb300.moe import Fp8MoELayer, quantize_expert_weights_fp8
    c = workloads.MOE_SMALL
    T, H, E, k, F = c["T"], c["H"], c["E"], c["k"], c["F"]
    r = routing(T, E, k, index=3)
    x = workloads.moe_activations(T, H, index=3)
    ids = r["topk_ids"]
    cnt = np.bincount(ids.reshape(-1), minlength=E)
    used = np.nonzero(cnt)[0]

    def token_of(e):
        return int(np.nonzero((ids == e).any(axis=1))[0][0])

    samples = sorted({0, T // 2, T - 1, token_of(int(cnt.argmax())), token_of(int(used[cnt[used].argmin()]))})
    experts = sorted({int(e) for t in samples for e in ids[t]})
    wl, host = [], {}
    for e in range(E):
        wgu, wd = workloads.moe_expert_weights(e, F, H, index=3, device="cuda")
        wl.append((wgu, wd))
        if e in experts:
            host[e] = (wgu.cpu(), wd.cpu())
    W = quantize_expert_weights_fp8([a for a, _ in wl], [b for _, b in wl])
    del wl
    layer = Fp8MoELayer(W, T, k)
    layer.capture(x.cuda(), logits=torch.from_numpy(r["logits"]).cuda())
    layer.replay()
    torch.cuda.synchronize()
    assert bs.device_status()[0] == 0
    assert np.array_equal(layer.topk_ids.cpu().numpy(), ids)
    _, w64 = oracle.moe_router(r["logits"], k)
    wts = layer.topk_w.cpu().numpy()
    assert np.allclose(wts, w64, rtol=ROUTER_RTOL, atol=0)
    _check_layer_stages(bs, layer, x, ids, wts, host, samples, F, H)
