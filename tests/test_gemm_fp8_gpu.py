"""FP8 e4m3 GEMM with 1x128 activation and 128x128 weight scales on the GPU vs
the FP64 oracle (codes and scales bit-exact first, then the GEMM within
|y - y_ref| <= 1e-3 S + 2^-8 |y_ref|, plus the tighter 1e-4 S diagnostic)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.helpers import gemm_errors, tight_errors

pytestmark = pytest.mark.gpu

# Decode shapes (fewer output tiles than SMs) run stream-K by default: the
# tiles' K blocks shared out over every SM, a tile's pieces summed by the last
# CTA to finish one (bs_gemm_args.fp8_stream_k = 1); 2 runs one CTA per tile.
# Every case runs both ways.
SCHEDULES = {"stream_k": 1, "per_tile": 2}


@pytest.fixture(autouse=True, params=sorted(SCHEDULES))
def fp8_schedule(request):
    import fp8_quantized_gemm_q4_gb300 as bs
    with bs.kernel_options(fp8_stream_k=SCHEDULES[request.param]):
        yield request.param


def run_fp8(bs, x, w, rows=None, out_dtype=torch.bfloat16, num_sms=0):
    xq, xs = bs.q8_quantize(x.cuda(), mode=bs.Q8_TOKEN)
    wq, ws = bs.q8_quantize(w.cuda(), mode=bs.Q8_BLOCK)
    y = bs.gemm_fp8(xq, xs, wq, ws, out_dtype=out_dtype, num_sms=num_sms)
    # the same call again, now as the weights-ready programmatic launch right
    # behind the activation quantizer: the same result bit for bit, and the
    # stream-K counters the first call left must have been reset to zero
    xq2, xs2 = bs.q8_quantize(x.cuda(), mode=bs.Q8_TOKEN)
    y2 = bs.gemm_fp8(xq2, xs2, wq, ws, out_dtype=out_dtype, num_sms=num_sms, weights_ready=True)
    torch.cuda.synchronize()
    assert bs.device_status()[0] == 0
    assert torch.equal(y, y2)
    M = x.shape[0]
    rows = np.arange(M) if rows is None else np.asarray(rows)
    oa, osa = oracle.q8_quantize(x[rows], rows_per_block=1)
    ob, osb = oracle.q8_quantize(w, rows_per_block=128)
    assert np.array_equal(xq.cpu().numpy()[rows], oa)
    assert np.array_equal(xs.cpu().numpy().T[rows], osa)
    assert np.array_equal(wq.cpu().numpy(), ob) and np.array_equal(ws.cpu().numpy(), osb)
    yr, s = oracle.gemm_fp8(oa, osa, ob, osb)
    yg = y.float().cpu().numpy()[rows]
    bf = out_dtype == torch.bfloat16
    ok, ratio, rel = gemm_errors(yg, yr, s, bf)
    tok, tratio = tight_errors(yg, yr, s, bf)
    return ok and tok, (ratio, rel, tratio)


@pytest.mark.parametrize("M", [1, 16, 64, 128])
def test_fp8_decode_sweep_full(cuda_lib, M):
    """The FP8 sweep workload (N = 7168, K = 4096, outlier channels), every row."""
    d = workloads.fp8_sweep(M)
    ok, info = run_fp8(cuda_lib, d["x"], d["w"])
    assert ok, info


def test_fp8_prefill_4096_sampled_rows(cuda_lib):
    d = workloads.fp8_sweep(4096)
    ok, info = run_fp8(cuda_lib, d["x"], d["w"], rows=[0, 1, 127, 128, 2047, 4000, 4095])
    assert ok, info


@pytest.mark.parametrize("M,N,K", [(3, 256, 256), (100, 384, 512), (300, 128, 128), (17, 640, 1024),
                                   (33, 128, 384), (200, 640, 256)])
def test_fp8_ragged(cuda_lib, M, N, K):
    g = torch.Generator().manual_seed(M + N + K)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    for dt in (torch.bfloat16, torch.float32):
        ok, info = run_fp8(cuda_lib, x, w, out_dtype=dt)
        assert ok, (dt, info)


@pytest.mark.parametrize("num_sms", [3, 57, 100, 151])
def test_fp8_stream_k_grid_sizes(cuda_lib, num_sms):
    """Decode shape on grids that cut the 56 x 32 K blocks unevenly: pieces
    of one tile spread over 1 to 4 CTAs, ranges that start and end inside
    tiles (3 SMs: fewer CTAs than tiles, whole tiles only)."""
    d = workloads.fp8_sweep(16)
    ok, info = run_fp8(cuda_lib, d["x"], d["w"], num_sms=num_sms)
    assert ok, info


def test_fp8_rejects_fp4_only_options(cuda_lib):
    bs = cuda_lib
    x = torch.randn(16, 128).to(torch.bfloat16).cuda()
    xq, xs = bs.q8_quantize(x)
    wq, ws = bs.q8_quantize(torch.randn(128, 128).to(torch.bfloat16).cuda(), mode=bs.Q8_BLOCK)
    g = bs._args(bs.FMT_FP8, xq, xs, wq, ws, 16, 128, 128, torch.empty(16, 128, dtype=torch.bfloat16, device="cuda"),
                 alpha=2.0)
    import ctypes
    assert bs.load().bs_gemm(ctypes.byref(g), None) == bs.BS_ERR_UNSUPPORTED
