"""FP4 GEMM on decode shapes (M <= 32): the swap-AB stream-K kernel against
the FP64 oracle, |y - y_ref| <= 1e-3 S + 2^-8 |y_ref| (bf16 output), plus the
tighter 1e-4 S diagnostic; the regular tile kernels (fp4_decode = 2) on the
same cases; repeated and weights-ready calls give identical results (the
stream-K counters return to zero)."""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import gemm_errors, tight_errors

pytestmark = pytest.mark.gpu


def _case(M, N, K, seed, wstd=0.02):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g) * wstd).to(torch.bfloat16)
    cs = (torch.rand(N, generator=g) + 0.5).float()
    bias = (torch.randn(N, generator=g) * 0.1).to(torch.bfloat16)
    return x, w, cs, bias


def _check(bs, x, w, cs, bias, out_dtype, alpha, decode, num_sms=0):
    K = x.shape[1]
    with bs.kernel_options(fp4_decode=1 if decode else 2):
        xq, xs, _ = bs.q4_quantize(x.cuda())
        wq, ws, _ = bs.q4_quantize(w.cuda())
        kw = dict(out_dtype=out_dtype, alpha=alpha, col_scale=None if cs is None else cs.cuda(),
                  bias=None if bias is None else bias.cuda(), num_sms=num_sms)
        y = bs.gemm_fp4(xq, xs, wq, ws, K, **kw)
        y2 = bs.gemm_fp4(xq, xs, wq, ws, K, weights_ready=True, **kw)
    torch.cuda.synchronize()
    assert bs.device_status()[0] == 0
    assert torch.equal(y, y2)
    oa, osa = oracle.q4_quantize(x)
    ob, osb = oracle.q4_quantize(w)
    yr, s = oracle.gemm_fp4(oa, osa, ob, osb, K, alpha=alpha, col_scale=cs, bias=bias)
    bf = out_dtype == torch.bfloat16
    yg = y.float().cpu().numpy()
    ok, ratio, rel = gemm_errors(yg, yr, s, bf)
    tok, tratio = tight_errors(yg, yr, s, bf)
    assert ok and tok, (ratio, rel, tratio)


@pytest.mark.parametrize("decode", [True, False], ids=["decode", "tiles"])
@pytest.mark.parametrize("M,N,K", [(1, 7168, 4096), (16, 7168, 4096), (5, 1024, 768), (17, 640, 256),
                                   (32, 2048, 2048), (3, 128, 256)])
def test_fp4_decode_bf16(cuda_lib, decode, M, N, K):
    x, w, _, _ = _case(M, N, K, M + N + K)
    _check(cuda_lib, x, w, None, None, torch.bfloat16, 1.0, decode)


@pytest.mark.parametrize("M", [1, 16, 32])
def test_fp4_decode_epilogue_fp32(cuda_lib, M):
    """alpha, per-column scale and bias in the decode kernel's epilogue, fp32 out."""
    x, w, cs, bias = _case(M, 1024, 1024, 7 * M)
    _check(cuda_lib, x, w, cs, bias, torch.float32, 0.75, True)


@pytest.mark.parametrize("num_sms", [3, 57, 100, 151])
def test_fp4_decode_grid_sizes(cuda_lib, num_sms):
    """56 tiles x 16 K stages cut unevenly over the grid (3 SMs: fewer CTAs
    than tiles, so each CTA takes a contiguous run of whole tiles)."""
    x, w, _, _ = _case(16, 7168, 4096, 5)
    _check(cuda_lib, x, w, None, None, torch.bfloat16, 1.0, True, num_sms=num_sms)


def test_fp4_decode_two_level_weights(cuda_lib):
    """Two-level weights on the decode kernel: the tensor scale read in its epilogue."""
    bs = cuda_lib
    x, w, _, _ = _case(8, 2048, 1024, 11)
    xq, xs, _ = bs.q4_quantize(x.cuda())
    wq, ws, wts = bs.q4_quantize_two_level(w.cuda())
    y = bs.gemm_fp4(xq, xs, wq, ws, 1024, b_tensor_scale=wts)
    torch.cuda.synchronize()
    oa, osa = oracle.q4_quantize(x)
    ob, osb, tb = oracle.q4_quantize_two_level(w)
    yr, s = oracle.gemm_fp4(oa, osa, ob, osb, 1024, alpha=tb)
    ok, ratio, rel = gemm_errors(y.float().cpu().numpy(), yr, s, True)
    assert ok, (ratio, rel)


@pytest.mark.parametrize("M,N,K", [(16, 1024, 1024), (16, 7168, 512), (32, 3968, 256)])
def test_fp4_decode_without_workspace(cuda_lib, M, N, K):
    """No caller workspace: whole tiles only, min(tiles, SMs) CTAs each taking a
    contiguous run balanced to within one tile (3968 = 31 tiles, a prime
    count); the result within tolerance of the oracle."""
    import ctypes
    bs = cuda_lib
    x, w, _, _ = _case(M, N, K, 3 * M + N + K)
    xq, xs, _ = bs.q4_quantize(x.cuda())
    wq, ws, _ = bs.q4_quantize(w.cuda())
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    g = bs._args(bs.FMT_FP4, xq, xs, wq, ws, M, N, K, y)
    assert g.workspace is None
    bs._check(bs.load().bs_gemm(ctypes.byref(g), bs._stream()))
    torch.cuda.synchronize()
    assert bs.device_status()[0] == 0
    oa, osa = oracle.q4_quantize(x)
    ob, osb = oracle.q4_quantize(w)
    yr, s = oracle.gemm_fp4(oa, osa, ob, osb, K)
    yg = y.float().cpu().numpy()
    ok, ratio, rel = gemm_errors(yg, yr, s, True)
    tok, tratio = tight_errors(yg, yr, s, True)
    assert ok and tok, (ratio, rel, tratio)
