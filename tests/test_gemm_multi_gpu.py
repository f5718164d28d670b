"""bs_gemm_multi: G GEMMs that share one activation (M <= 32), in one launch,
on the GPU -- block-scaled FP8 and FP4 through the decode kernel.  Every
product must equal the oracle's FP64 GEMM of the same codes within the GEMM
tolerance (|y - y_ref| <= 1e-3 S + 2^-8 |y_ref|, plus the tighter 1e-4 S
diagnostic).  FP8 products also equal, bit for bit, the single-weight bs_gemm
result wherever both run whole tiles (each output tile accumulated by one CTA
in K order); FP4 products run stream-K over all products' K stages, so their
pieces differ from a single call's and only G = 1 is compared bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.helpers import gemm_errors, tight_errors

pytestmark = pytest.mark.gpu


def weight_sets(G, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    return [(torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16) for _ in range(G)]


def quantized(bs, x, ws):
    xq, xs = bs.q8_quantize(x.cuda(), mode=bs.Q8_TOKEN)
    wqs = [bs.q8_quantize(w.cuda(), mode=bs.Q8_BLOCK) for w in ws]
    return xq, xs, wqs


def check_vs_oracle(x, w, xq, xs, wq, wsc, y, rows=None):
    """The GPU's codes and scales equal the oracle's; y within tolerance."""
    M = x.shape[0]
    rows = np.arange(M) if rows is None else np.asarray(rows)
    oa, osa = oracle.q8_quantize(x[rows], rows_per_block=1)
    ob, osb = oracle.q8_quantize(w, rows_per_block=128)
    assert np.array_equal(xq.cpu().numpy()[rows], oa)
    assert np.array_equal(xs.cpu().numpy().T[rows], osa)
    assert np.array_equal(wq.cpu().numpy(), ob) and np.array_equal(wsc.cpu().numpy(), osb)
    yr, s = oracle.gemm_fp8(oa, osa, ob, osb)
    yg = y.float().cpu().numpy()[rows]
    bf = y.dtype == torch.bfloat16
    ok, ratio, rel = gemm_errors(yg, yr, s, bf)
    tok, tratio = tight_errors(yg, yr, s, bf)
    return ok and tok, (ratio, rel, tratio)


@pytest.mark.parametrize("M,N,K,G", [(1, 1024, 1024, 3), (16, 384, 512, 8), (32, 1024, 256, 2),
                                     (7, 128, 128, 5)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_multi_whole_tiles_equal_single_calls(cuda_lib, M, N, K, G, out_dtype):
    """One CTA per tile on both sides: each product bit-identical to bs_gemm
    on its own weights, and within tolerance of the oracle."""
    bs = cuda_lib
    g = torch.Generator().manual_seed(M * 1000 + N + K + G)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    ws = weight_sets(G, N, K, seed=G * 7 + M)
    xq, xs, wqs = quantized(bs, x, ws)
    with bs.kernel_options(fp8_stream_k=2):
        ys = bs.gemm_fp8_multi(xq, xs, wqs, out_dtype=out_dtype)
        singles = [bs.gemm_fp8(xq, xs, wq, wsc, out_dtype=out_dtype) for wq, wsc in wqs]
    torch.cuda.synchronize()
    assert bs.device_status()[0] == 0
    for i, (y, y1) in enumerate(zip(ys, singles)):
        assert torch.equal(y, y1), i
    for i in (0, G - 1):
        ok, info = check_vs_oracle(x, ws[i], xq, xs, *wqs[i], ys[i])
        assert ok, (i, info)


@pytest.mark.parametrize("num_sms", [0, 5, 77])
def test_multi_stream_k_vs_oracle(cuda_lib, num_sms):
    """Fewer tiles than SMs over all products (5 x 5 tiles): the products' K
    blocks shared out by stream-K; every product within tolerance of the
    oracle, the call repeatable bit for bit (tile counters back at zero) and
    equal when launched as the weights-ready dependent of the quantizer."""
    bs = cuda_lib
    M, N, K, G = 16, 640, 2048, 5
    g = torch.Generator().manual_seed(11)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    ws = weight_sets(G, N, K, seed=12)
    xq, xs, wqs = quantized(bs, x, ws)
    y1 = bs.gemm_fp8_multi(xq, xs, wqs, num_sms=num_sms)
    y1 = [y.clone() for y in y1]
    xq2, xs2 = bs.q8_quantize(x.cuda(), mode=bs.Q8_TOKEN)
    y2 = bs.gemm_fp8_multi(xq2, xs2, wqs, num_sms=num_sms, weights_ready=True)
    torch.cuda.synchronize()
    assert bs.device_status()[0] == 0
    for a, b in zip(y1, y2):
        assert torch.equal(a, b)
    for i in range(G):
        ok, info = check_vs_oracle(x, ws[i], xq, xs, *wqs[i], y1[i])
        assert ok, (i, info)


def test_multi_single_product_is_bs_gemm(cuda_lib):
    bs = cuda_lib
    d = workloads.fp8_sweep(16, N=1024, K=1024)
    xq, xs, wqs = quantized(bs, d["x"], [d["w"]])
    y = bs.gemm_fp8_multi(xq, xs, wqs)[0]
    y1 = bs.gemm_fp8(xq, xs, *wqs[0])
    torch.cuda.synchronize()
    assert torch.equal(y, y1)


def test_multi_decode_full_size(cuda_lib):
    """The decode projections at full size: M = 16 tokens of the FP8 sweep
    (outlier channels) against 8 weight sets of [7168, 4096] -- 448 tiles, one
    grid.  Every product bit-identical to its whole-tile single call; the
    first and last against the oracle on every row."""
    bs = cuda_lib
    G = 8
    d = workloads.fp8_sweep(16)
    ws = [d["w"]] + weight_sets(G - 1, 7168, 4096, seed=99)
    xq, xs, wqs = quantized(bs, d["x"], ws)
    ys = bs.gemm_fp8_multi(xq, xs, wqs)
    with bs.kernel_options(fp8_stream_k=2):
        singles = [bs.gemm_fp8(xq, xs, wq, wsc) for wq, wsc in wqs]
    torch.cuda.synchronize()
    assert bs.device_status()[0] == 0
    for i, (y, y1) in enumerate(zip(ys, singles)):
        assert torch.equal(y, y1), i
    for i in (0, G - 1):
        ok, info = check_vs_oracle(d["x"], ws[i], xq, xs, *wqs[i], ys[i])
        assert ok, (i, info)


def test_multi_rejects(cuda_lib):
    bs = cuda_lib
    x = torch.randn(40, 256).to(torch.bfloat16).cuda()
    xq, xs = bs.q8_quantize(x)
    wq, wsc = bs.q8_quantize(torch.randn(128, 256).to(torch.bfloat16).cuda(), mode=bs.Q8_BLOCK)
    with pytest.raises(bs.BSError) as e:
        bs.gemm_fp8_multi(xq, xs, [(wq, wsc)] * 2)              # M = 40 > 32
    assert e.value.status == bs.BS_ERR_UNSUPPORTED
    with pytest.raises(bs.BSError) as e:
        bs.gemm_fp8_multi(xq[:16], xs, [(wq, wsc)] * 9)         # G = 9
    assert e.value.status == bs.BS_ERR_INVALID


# ----------------------------------------------------------------------------- FP4


def fp4_inputs(bs, M, N, K, G, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    ws = weight_sets(G, N, K, seed + 1)
    xq, xs, _ = bs.q4_quantize(x.cuda())
    wqs = [bs.q4_quantize(w.cuda())[:2] for w in ws]
    return x, ws, xq, xs, wqs


def check_fp4_vs_oracle(x, w, y, K, alpha=1.0):
    oa, osa = oracle.q4_quantize(x)
    ob, osb = oracle.q4_quantize(w)
    yr, s = oracle.gemm_fp4(oa, osa, ob, osb, K, alpha=alpha)
    bf = y.dtype == torch.bfloat16
    yg = y.float().cpu().numpy()
    ok, ratio, rel = gemm_errors(yg, yr, s, bf)
    tok, tratio = tight_errors(yg, yr, s, bf)
    return ok and tok, (ratio, rel, tratio)


@pytest.mark.parametrize("M,N,K,G", [(1, 1024, 1024, 3), (16, 384, 2048, 8), (32, 640, 256, 5), (5, 128, 768, 2)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_fp4_multi_vs_oracle(cuda_lib, M, N, K, G, out_dtype):
    """Every product within tolerance of the oracle (alpha 0.75 on all of
    them); the call repeatable bit for bit and equal as the weights-ready
    dependent of the activation quantizer (stream-K counters back at zero)."""
    bs = cuda_lib
    x, ws, xq, xs, wqs = fp4_inputs(bs, M, N, K, G, seed=M * 31 + N + K + G)
    y1 = [y.clone() for y in bs.gemm_fp4_multi(xq, xs, wqs, K, out_dtype=out_dtype, alpha=0.75)]
    xq2, xs2, _ = bs.q4_quantize(x.cuda())
    y2 = bs.gemm_fp4_multi(xq2, xs2, wqs, K, out_dtype=out_dtype, alpha=0.75, weights_ready=True)
    torch.cuda.synchronize()
    assert bs.device_status()[0] == 0
    for a, b in zip(y1, y2):
        assert torch.equal(a, b)
    for i in range(G):
        ok, info = check_fp4_vs_oracle(x, ws[i], y1[i], K, alpha=0.75)
        assert ok, (i, info)


def test_fp4_multi_single_product_is_bs_gemm(cuda_lib):
    bs = cuda_lib
    x, ws, xq, xs, wqs = fp4_inputs(bs, 16, 1024, 1024, 1, seed=5)
    y = bs.gemm_fp4_multi(xq, xs, wqs, 1024)[0]
    y1 = bs.gemm_fp4(xq, xs, *wqs[0], 1024)
    torch.cuda.synchronize()
    assert torch.equal(y, y1)


def test_fp4_multi_decode_full_size(cuda_lib):
    """8 FP4 weight sets of [7168, 4096] against M = 16 tokens in one launch:
    the first and last products against the oracle on every row; every
    product within a tight bound of its own single-weight call (the same
    arithmetic up to the stream-K split of the fp32 sum)."""
    bs = cuda_lib
    G, M, N, K = 8, 16, 7168, 4096
    x, ws, xq, xs, wqs = fp4_inputs(bs, M, N, K, G, seed=77)
    ys = bs.gemm_fp4_multi(xq, xs, wqs, K, out_dtype=torch.float32)
    singles = [bs.gemm_fp4(xq, xs, wq, wsc, K, out_dtype=torch.float32) for wq, wsc in wqs]
    torch.cuda.synchronize()
    assert bs.device_status()[0] == 0
    for i, (y, y1) in enumerate(zip(ys, singles)):
        scale = y1.abs().max().item()
        assert torch.allclose(y, y1, rtol=1e-5, atol=1e-5 * scale), i
    for i in (0, G - 1):
        ok, info = check_fp4_vs_oracle(x, ws[i], ys[i], K)
        assert ok, (i, info)
