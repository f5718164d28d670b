"""bs_gemm_multi: G block-scaled FP8 GEMMs that share one activation, in one
launch, on the GPU.  Every product must equal the oracle's FP64 GEMM of the
same codes within the FP8 GEMM tolerance (|y - y_ref| <= 1e-3 S + 2^-8
|y_ref|, plus the tighter 1e-4 S diagnostic), and -- where both run whole
tiles, so that each output tile is accumulated by one CTA in K order -- be bit
for bit the single-weight bs_gemm result for that weight set."""
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
