"""Grouped FP4 MoE path on the GPU vs the FP64 oracle.

Dispatch is integer work: bit-exact.  The grouped GEMMs are checked in
stages, because re-quantizing a slightly different h may legitimately flip a
code: (1) h against the oracle's SwiGLU of the oracle GEMMs on the GPU's own
activation codes; (2) the GPU's re-quantized h bit-exact against the oracle
re-quantizing the GPU's h; (3) the combined output against the oracle fed
with the GPU's quantized h.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.conftest import read_golden
from tests.helpers import gemm_errors, sf_rowmajor, routing

pytestmark = pytest.mark.gpu

# Router weights: the GPU takes exp(l_j - l_0) in fp32 (one rounding of the
# difference, scaled by |l_j - l_0| <= 32 here, plus expf's <= 2 ulp), sums k
# <= 32 terms and divides once: relative error below (32 + 2 + 32 + 1) 2^-24
# < 4e-6 of the FP64 softmax.
ROUTER_RTOL = 4e-6


@pytest.fixture(params=["pair", "pair_whole", "one_cta"])
def fp4_kernel(request):
    """Grouped GEMMs on CTA pairs with the small experts (<= 128 rows) in a
    second one-CTA launch (default), on CTA pairs alone, or on the one-CTA
    kernel alone (bs_gemm_args.fp4_kernel / fp4_small_experts)."""
    import fp8_quantized_gemm_q4_gb300 as bs
    with bs.kernel_options(fp4_kernel=1 if request.param == "one_cta" else 2,
                           fp4_small_experts=2 if request.param == "pair_whole" else 1):
        yield request.param


def test_dispatch_hand_case(cuda_lib):
    bs = cuda_lib
    gold = {r[0]: [int(v) for v in r[1:]] for r in read_golden("moe_dispatch_2x8.txt")}
    ids = torch.tensor([[t % 2, 1 - t % 2] for t in range(8)], dtype=torch.int32)
    w = torch.full((8, 2), 0.5)
    d = bs.moe_dispatch(ids.cuda(), w.cuda(), E=2)
    torch.cuda.synchronize()
    assert d["counts"].tolist() == gold["counts"]
    assert d["offsets"].tolist() == gold["offsets"]
    por = d["pair_of_row"].cpu()
    assert por[0:8].tolist() == gold["expert0_pairs"] and por[128:136].tolist() == gold["expert1_pairs"]
    assert (por[8:128] == -1).all() and (por[136:] == -1).all()


@pytest.mark.parametrize("T,E,k", [(1, 4, 2), (300, 9, 4), (4096, 64, 8), (16384, 256, 8)])
def test_dispatch_bit_exact(cuda_lib, T, E, k):
    bs = cuda_lib
    r = routing(T, E, k)
    ids, w = torch.from_numpy(r["topk_ids"]), torch.from_numpy(r["topk_w"])
    d = bs.moe_dispatch(ids.cuda(), w.cuda(), E=E)
    torch.cuda.synchronize()
    counts, offsets, por = oracle.moe_dispatch(r["topk_ids"], E)
    assert np.array_equal(d["counts"].cpu().numpy(), counts)
    assert np.array_equal(d["offsets"].cpu().numpy(), offsets)
    gp = d["pair_of_row"].cpu().numpy()
    assert np.array_equal(gp[:offsets[E]], por)
    assert np.all(gp[offsets[E]:] == -1)
    tok = d["token_of"].cpu().numpy()
    wt = d["weight_of"].cpu().numpy()
    real = gp >= 0
    assert np.array_equal(tok[real], gp[real] // k) and np.all(tok[~real] == -1)
    assert np.array_equal(wt[real], r["topk_w"].reshape(-1)[gp[real]]) and np.all(wt[~real] == 0)
    assert bs.device_status()[0] == 0


def _small_moe(T=200, H=256, F=128, E=5, k=2, seed=3):
    r = routing(T, E, k, index=seed)
    x = workloads.moe_activations(T, H, index=seed)
    ws = [workloads.moe_expert_weights(e, F, H, index=seed) for e in range(E)]
    return r, x, ws


@pytest.mark.parametrize("T,H,F,E,k,chunk", [(200, 256, 128, 5, 2, 0), (1000, 512, 256, 8, 4, 0),
                                             (64, 256, 128, 16, 8, 0), (300, 1024, 256, 6, 2, 1),
                                             (300, 1024, 256, 6, 2, 3)])
@pytest.mark.parametrize("combine", ["rows", "atomic"])
def test_grouped_layer_staged(cuda_lib, fp4_kernel, combine, T, H, F, E, k, chunk):
    """combine="rows": weighted fp32 rows, then a slot-order sum per token;
    "atomic": fp32 reductions into out32.  chunk > 0 (atomic): the down GEMM
    walks column chunks of that many 256-wide blocks.  The stages run on the
    separate-h path (bf16 h visible); the default path, h quantized in the
    gate/up epilogue, must then give the same codes, scales and output."""
    bs = cuda_lib
    from fp8_quantized_gemm_q4_gb300.moe import MoELayer, quantize_expert_weights
    r, x, ws = _small_moe(T, H, F, E, k)
    W = quantize_expert_weights([a for a, _ in ws], [b for _, b in ws])
    layer = MoELayer(W, T, k, combine=combine, h_quant="separate")
    if chunk:
        layer.combine_chunk = chunk
    out = layer.forward(x.cuda(), torch.from_numpy(r["topk_ids"]).cuda(), torch.from_numpy(r["topk_w"]).cuda())
    torch.cuda.synchronize()
    assert bs.device_status()[0] == 0
    counts, offsets, por = oracle.moe_dispatch(r["topk_ids"], E)
    rows = offsets[E]
    # activation codes of the routed rows
    xq = layer.xq.cpu().numpy()[:rows]
    real = por >= 0
    oa, osa = oracle.q4_quantize(x[por[real] // k])
    assert np.array_equal(xq[real], oa)
    assert np.array_equal(sf_rowmajor(layer.xs.cpu().numpy(), rows, H)[real], osa)
    # stage 1: h from the oracle GEMMs on the GPU codes
    h = layer.h.float().cpu().numpy()[:rows]
    assert np.all(h[~real] == 0)
    wgu = [oracle.q4_quantize(a) for a, _ in ws]
    wd = [oracle.q4_quantize(b) for _, b in ws]
    for e in range(E):
        seg = np.arange(offsets[e], offsets[e] + counts[e])
        if len(seg) == 0:
            continue
        gu, s_gu = oracle.gemm_fp4(xq[seg], sf_rowmajor(layer.xs.cpu().numpy(), rows, H)[seg], wgu[e][0], wgu[e][1], H)
        g, u = gu[:, :F], gu[:, F:]
        h_ref = oracle.swiglu(g, u)
        # error of silu(g) u from |g - g_ref| <= 1e-3 S_g and |u - u_ref| <= 1e-3 S_u, plus bf16 rounding
        sig = 1.0 / (1.0 + np.exp(-g))
        dsilu = np.abs(sig * (1 + g * (1 - sig)))
        bound = 1e-3 * (dsilu * np.abs(u) * s_gu[:, :F] + np.abs(g * sig) * s_gu[:, F:]) + 2.0 ** -8 * np.abs(h_ref)
        assert np.all(np.abs(h[seg] - h_ref) <= bound + 1e-30), e
    # stage 2: re-quantized h bit-exact against the oracle on the GPU's h
    hq = layer.hq.cpu().numpy()[:rows]
    ohq, ohs = oracle.q4_quantize(layer.h[:rows].cpu())
    assert np.array_equal(hq, ohq)
    assert np.array_equal(sf_rowmajor(layer.hs.cpu().numpy(), rows, F), ohs)
    # stage 3: combine against the oracle down GEMM on the GPU's quantized h
    ref = np.zeros((T, H))
    S = np.zeros((T, H))
    wflat = r["topk_w"].reshape(-1).astype(np.float64)
    for e in range(E):
        seg = np.arange(offsets[e], offsets[e] + counts[e])
        if len(seg) == 0:
            continue
        y, sy = oracle.gemm_fp4(hq[seg], ohs[seg], wd[e][0], wd[e][1], F)
        pairs = por[seg]
        np.add.at(ref, pairs // k, wflat[pairs][:, None] * y)
        np.add.at(S, pairs // k, np.abs(wflat[pairs][:, None]) * sy)
    ok, ratio, rel = gemm_errors(out.float().cpu().numpy(), ref, S, True)
    assert ok, (ratio, rel)
    # the fused path: h quantized in the gate/up epilogue
    fused = MoELayer(W, T, k, combine=combine)
    if chunk:
        fused.combine_chunk = chunk
    assert fused.h_quant == "fused" and fused.h is None
    out_f = fused.forward(x.cuda(), torch.from_numpy(r["topk_ids"]).cuda(), torch.from_numpy(r["topk_w"]).cuda())
    torch.cuda.synchronize()
    assert bs.device_status()[0] == 0
    assert np.array_equal(fused.hq.cpu().numpy()[:rows], hq)
    assert np.array_equal(sf_rowmajor(fused.hs.cpu().numpy(), rows, F), sf_rowmajor(layer.hs.cpu().numpy(), rows, F))
    if combine == "rows":  # the atomic combine's reduction order may differ between runs
        assert torch.equal(out_f.view(torch.int16), out.view(torch.int16))
    if combine == "atomic":
        # out32 was reset by the finalize step
        assert float(layer.out32.abs().max()) == 0.0
    else:
        # a written padding row (one sharing a 32-row box with real rows) is zero
        yrows = layer.yrows[:rows].cpu().numpy()
        shared = np.zeros(rows, dtype=bool)
        for b0 in range(0, rows, 32):
            shared[b0:b0 + 32] = real[b0:b0 + 32].any()
        assert np.all(yrows[~real & shared] == 0)


@pytest.mark.parametrize("T,k,H,n_rows,drop", [(1, 1, 8, 128, 0), (300, 4, 264, 1536, 7), (1000, 8, 1024, 8320, 31),
                                               (50, 11, 64, 768, 3)])
def test_combine_bit_exact(cuda_lib, T, k, H, n_rows, drop):
    """bs_moe_combine against a float32 sum in slot order (absent slots add +0)
    rounded once to bf16: bit-exact.  Pairs are placed on random rows; `drop`
    pairs have no row (as for out-of-range expert ids)."""
    bs = cuda_lib
    rng = np.random.default_rng(T * 1000 + k)
    P = T * k
    rows_of = rng.permutation(n_rows)[:P].astype(np.int32)
    dropped = rng.choice(P, size=drop, replace=False) if drop else np.zeros(0, dtype=np.int64)
    pair_of_row = np.full(n_rows, -1, dtype=np.int32)
    keep = np.setdiff1d(np.arange(P), dropped)
    pair_of_row[rows_of[keep]] = keep
    rows = rng.standard_normal((n_rows, H)).astype(np.float32)
    acc = np.zeros((T, H), dtype=np.float32)
    for j in range(k):
        p = np.arange(T) * k + j
        r = np.where(np.isin(p, dropped), -1, rows_of[p])
        add = np.where((r >= 0)[:, None], rows[np.maximum(r, 0)], np.float32(0.0))
        acc = (acc + add).astype(np.float32)
    ref = torch.from_numpy(acc).to(torch.bfloat16)
    out = bs.moe_combine(torch.from_numpy(rows).cuda(), torch.from_numpy(pair_of_row).cuda(), T, k)
    out2 = bs.moe_combine(torch.from_numpy(rows).cuda(), torch.from_numpy(pair_of_row).cuda(), T, k)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu().view(torch.int16), ref.view(torch.int16))
    assert torch.equal(out2.cpu().view(torch.int16), ref.view(torch.int16))


def test_layer_end_to_end_report(cuda_lib):
    """End to end against the oracle's own layer (its own h and re-quantization):
    looser, reported, with a bound that allows re-quantization flips."""
    bs = cuda_lib
    from fp8_quantized_gemm_q4_gb300.moe import MoELayer, quantize_expert_weights
    T, H, F, E, k = 64, 256, 128, 4, 2
    r, x, ws = _small_moe(T, H, F, E, k)
    W = quantize_expert_weights([a for a, _ in ws], [b for _, b in ws])
    out = MoELayer(W, T, k).forward(x.cuda(), torch.from_numpy(r["topk_ids"]).cuda(),
                                    torch.from_numpy(r["topk_w"]).cuda())
    torch.cuda.synchronize()
    wgu = [oracle.q4_quantize(a) for a, _ in ws]
    wd = [oracle.q4_quantize(b) for _, b in ws]
    ref = oracle.moe_layer(x, r["topk_ids"], r["topk_w"], [c for c, _ in wgu], [s for _, s in wgu],
                           [c for c, _ in wd], [s for _, s in wd], F=F)["out"]
    o = out.float().cpu().numpy()
    rel = np.abs(o - ref).max() / np.abs(ref).max()
    print(f"end-to-end MoE max |err| / max |ref| = {rel:.3g}")
    assert rel < 0.05
    assert bs.device_status()[0] == 0


def _sf_rows(sf, rows, K):
    """Scale bytes of the given rows from the MMA layout ([len(rows), K/16])."""
    sf = np.asarray(sf).reshape(-1)
    r = np.asarray(rows)[:, None]
    g = np.arange(K // 16)[None, :]
    off = ((r // 128) * (K // 64) + g // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + g % 4
    return sf[off]


@pytest.mark.parametrize("cfg,index", [("MOE_SMALL", 3), ("MOE_LARGE", 4)])
def test_full_size_layer_sampled_tokens(cuda_lib, cfg, index):
    """The benchmark's MoE layers at full size, through the same layer object
    the bench times (two-pass combine, CTA pairs), checked on sampled tokens in
    the same stages as the small-shape test: routed activation codes
    bit-exact, h against the oracle's SwiGLU of its GEMMs on the GPU's codes,
    re-quantized h bit-exact, and the combined output against the oracle's
    down GEMMs on the GPU's quantized h."""
    bs = cuda_lib
    from fp8_quantized_gemm_q4_gb300.moe import MoELayer, MoEWeights
    c = getattr(workloads, cfg)
    T, H, E, k, F = c["T"], c["H"], c["E"], c["k"], c["F"]
    r = routing(T, E, k, index=index)
    x = workloads.moe_activations(T, H, index=index)
    ids = r["topk_ids"]
    # tokens: first, middle, last; one routed to the most loaded expert; one
    # routed to an expert of at most 128 rows (served by the one-CTA launch);
    # the last token of an expert whose last 256-row pair tile is partly full
    cnt = np.bincount(ids.reshape(-1), minlength=E)
    heavy = int(cnt.argmax())
    small = [e for e in range(E) if 1 <= cnt[e] <= 128]
    partial = [e for e in range(E) if cnt[e] > 128 and cnt[e] % 256 != 0]
    assert small and partial

    def token_of(e, last=False):
        return int(np.nonzero((ids == e).any(axis=1))[0][-1 if last else 0])

    samples = sorted({0, T // 2, T - 1, token_of(heavy), token_of(small[0]), token_of(partial[0], last=True)})
    experts = sorted({int(e) for t in samples for e in ids[t]})
    F2 = 2 * F
    wgu_codes = torch.empty((E * F2, H // 2), dtype=torch.uint8, device="cuda")
    wgu_sf = torch.empty(bs.sf_bytes(E * F2, H), dtype=torch.uint8, device="cuda")
    wd_codes = torch.empty((E * H, F // 2), dtype=torch.uint8, device="cuda")
    wd_sf = torch.empty(bs.sf_bytes(E * H, F), dtype=torch.uint8, device="cuda")
    pg, pd = bs.sf_bytes(F2, H), bs.sf_bytes(H, F)
    host_w = {}
    for e in range(E):
        wgu, wd = workloads.moe_expert_weights(e, F, H, index=index, device="cuda")
        bs.q4_quantize(wgu, out=(wgu_codes[e * F2:(e + 1) * F2], wgu_sf[e * pg:(e + 1) * pg], None))
        bs.q4_quantize(wd, out=(wd_codes[e * H:(e + 1) * H], wd_sf[e * pd:(e + 1) * pd], None))
        if e in experts:
            host_w[e] = (wgu.cpu(), wd.cpu())
        del wgu, wd
    Wt = MoEWeights(E, H, F, wgu_codes, wgu_sf, wd_codes, wd_sf)
    layer = MoELayer(Wt, T, k, h_quant="separate")  # bf16 h visible for the stages
    # from the router's logits, as the bench runs it: the GPU router's experts
    # equal the oracle's, its weights are within the fp32 softmax's rounding
    out = layer.forward_logits(x.cuda(), torch.from_numpy(r["logits"]).cuda())
    torch.cuda.synchronize()
    assert bs.device_status()[0] == 0
    assert np.array_equal(layer.topk_ids.cpu().numpy(), ids)
    _, w64 = oracle.moe_router(r["logits"], k)
    wts = layer.topk_w.cpu().numpy()
    assert np.allclose(wts, w64, rtol=ROUTER_RTOL, atol=0)
    # the bench's path (h quantized in the gate/up epilogue): same codes and
    # scales on every row of the expert segments, same output bit for bit
    fused = MoELayer(Wt, T, k)
    out_f = fused.forward_logits(x.cuda(), torch.from_numpy(r["logits"]).cuda())
    torch.cuda.synchronize()
    assert bs.device_status()[0] == 0
    seg_rows = int(fused.disp["offsets"][E])
    assert torch.equal(fused.hq[:seg_rows], layer.hq[:seg_rows])
    nblk = (seg_rows + 127) // 128
    per_blk = bs.sf_bytes(128, F)
    assert torch.equal(fused.hs[:nblk * per_blk], layer.hs[:nblk * per_blk])
    assert torch.equal(out_f.view(torch.int16), out.view(torch.int16))
    del fused
    rop = layer.row_of_pair.cpu().numpy()
    rows = np.array([rop[t * k + j] for t in samples for j in range(k)])
    assert np.all(rows >= 0)
    xq = layer.xq[torch.from_numpy(rows).cuda().long()].cpu().numpy()
    xs = _sf_rows(layer.xs.cpu().numpy(), rows, H)
    oa, osa = oracle.q4_quantize(x[[t for t in samples for _ in range(k)]])
    assert np.array_equal(xq, oa) and np.array_equal(xs, osa)
    h = layer.h[torch.from_numpy(rows).cuda().long()].float().cpu().numpy()
    hq = layer.hq[torch.from_numpy(rows).cuda().long()].cpu().numpy()
    hs = _sf_rows(layer.hs.cpu().numpy(), rows, F)
    ohq, ohs = oracle.q4_quantize(layer.h[torch.from_numpy(rows).cuda().long()].cpu())
    assert np.array_equal(hq, ohq) and np.array_equal(hs, ohs)
    oq = {e: (oracle.q4_quantize(host_w[e][0]), oracle.q4_quantize(host_w[e][1])) for e in experts}
    got = out.float().cpu().numpy()
    for i, t in enumerate(samples):
        ref = np.zeros(H)
        S = np.zeros(H)
        for j in range(k):
            n = i * k + j
            e = int(ids[t, j])
            (gu_c, gu_s), (d_c, d_s) = oq[e]
            gu, s_gu = oracle.gemm_fp4(xq[n:n + 1], xs[n:n + 1], gu_c, gu_s, H)
            g_, u_ = gu[:, :F], gu[:, F:]
            h_ref = oracle.swiglu(g_, u_)
            sig = 1.0 / (1.0 + np.exp(-g_))
            dsilu = np.abs(sig * (1 + g_ * (1 - sig)))
            bound = 1e-3 * (dsilu * np.abs(u_) * s_gu[:, :F] + np.abs(g_ * sig) * s_gu[:, F:]) + 2.0 ** -8 * np.abs(h_ref)
            assert np.all(np.abs(h[n:n + 1] - h_ref) <= bound + 1e-30), (t, j)
            y, sy = oracle.gemm_fp4(hq[n:n + 1], hs[n:n + 1], d_c, d_s, F)
            wgt = float(wts[t, j])
            ref += wgt * y[0]
            S += abs(wgt) * sy[0]
        ok, ratio, rel = gemm_errors(got[t:t + 1], ref[None], S[None], True)
        assert ok, (t, ratio, rel)


def test_layer_graph_replay_matches_forward(cuda_lib):
    """The layer captured as one CUDA graph: replays give the eager forward's
    output bit for bit (the combine is deterministic), also after new
    activations are copied in."""
    from fp8_quantized_gemm_q4_gb300.moe import MoELayer, quantize_expert_weights
    T, H, F, E, k = 300, 512, 256, 6, 4
    r, x, ws = _small_moe(T, H, F, E, k)
    W = quantize_expert_weights([a for a, _ in ws], [b for _, b in ws])
    ids = torch.from_numpy(r["topk_ids"]).cuda()
    w = torch.from_numpy(r["topk_w"]).cuda()
    xd = x.cuda()
    ref = MoELayer(W, T, k).forward(xd, ids, w).clone()
    x2 = (x.float() * 0.5 + 0.125).to(torch.bfloat16).cuda()
    ref2 = MoELayer(W, T, k).forward(x2, ids, w).clone()
    layer = MoELayer(W, T, k)
    layer.capture(xd, ids, w)
    out1 = layer.replay().clone()
    out2 = layer.replay(x2).clone()
    out3 = layer.replay(xd).clone()
    torch.cuda.synchronize()
    assert cuda_lib.device_status()[0] == 0
    assert torch.equal(out1, ref) and torch.equal(out2, ref2) and torch.equal(out3, ref)


@pytest.mark.parametrize("T,E,k,ties", [(4096, 64, 8, False), (16384, 256, 8, False), (37, 13, 13, True),
                                        (300, 1024, 32, False), (5, 33, 1, True), (700, 256, 8, True),
                                        (0, 64, 8, False)])
def test_router_topk_matches_oracle(cuda_lib, T, E, k, ties):
    """Top-k experts bit-exact against the oracle (the same fp32 logits decide
    both), weights within ROUTER_RTOL of its FP64 softmax.  `ties`: logits
    rounded to one decimal, so equal logits are common and the lower expert
    id must win every tie."""
    bs = cuda_lib
    logits = workloads.moe_logits(max(T, 1), E, index=T + E)[:T]
    if ties:
        logits = np.round(logits, 1).astype(np.float32)
    ids, w = bs.moe_router_topk(torch.from_numpy(logits).cuda(), k)
    torch.cuda.synchronize()
    oids, ow = oracle.moe_router(logits, k)
    assert np.array_equal(ids.cpu().numpy(), oids)
    assert np.allclose(w.cpu().numpy(), ow, rtol=ROUTER_RTOL, atol=0)


def test_router_rejects_bad_sizes(cuda_lib):
    bs = cuda_lib
    lg = torch.zeros((4, 8), device="cuda")
    for k in (0, 9):
        with pytest.raises(bs.BSError) as e:
            bs.moe_router_topk(lg, k)
        assert e.value.status == bs.BS_ERR_INVALID
    with pytest.raises(bs.BSError):
        bs.moe_router_topk(torch.zeros((4, 40), device="cuda"), 33)   # k > 32
