"""Format variants on the GPU against the oracle ("Tencent AI Infra interview
notes": the scale-granularity table and W8A8 SmoothQuant).

Two-level FP4: tensor amax, codes, group scales and the power-of-two tensor
scale bit-exact; the dense GEMM on two-level operands within the GEMM
tolerance (|y - y_ref| <= 1e-3 S + 2^-8 |y_ref| for bf16 output).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.helpers import gemm_errors, sf_rowmajor, tight_errors

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K,dtype,std", [(1, 64, torch.float32, 1.0), (300, 512, torch.bfloat16, 0.02),
                                           (128, 1024, torch.float32, 3.0e3), (77, 256, torch.bfloat16, 1e-30),
                                           (64, 128, torch.float32, 1e-41), (40, 192, torch.bfloat16, 0.0)])
def test_q4_two_level_bit_exact(cuda_lib, M, K, dtype, std):
    """std 1e-41: fp32 subnormal input, whose tensor scale 2^e lies below the
    fp32 normal range (the quantizer then scales with ldexpf); std 0: a zero
    tensor (e = 0)."""
    bs = cuda_lib
    g = torch.Generator().manual_seed(M + K)
    x = (torch.randn(M, K, generator=g, dtype=torch.float64) * std).to(dtype)
    xd = x.cuda()
    amax = bs.tensor_amax(xd)
    codes, sf, ts = bs.q4_quantize_two_level(xd, amax=amax)
    torch.cuda.synchronize()
    xf = x.float().numpy()
    assert amax.item() == np.float32(np.abs(xf).max())
    oc, os_, ots = oracle.q4_quantize_two_level(xf)
    assert ts.item() == ots
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(sf_rowmajor(sf.cpu().numpy(), M, K), os_)


@pytest.mark.parametrize("kernel", [1, 2], ids=["one_cta", "pair"])
@pytest.mark.parametrize("M,N,K", [(256, 512, 1024), (300, 384, 512), (2048, 2048, 2048)])
def test_gemm_fp4_two_level(cuda_lib, kernel, M, N, K):
    """Weights N(0, 0.02) and activations N(0, 1), both two-level; the GEMM
    multiplies by the two tensor scales read from device memory."""
    bs = cuda_lib
    d = workloads.dense_lowrank(M=M, N=N, K=K, lowrank=False, bias=False)
    w = (d["w"].float() * 0.02).to(torch.bfloat16)
    with bs.kernel_options(fp4_kernel=kernel):
        xq, xs, xts = bs.q4_quantize_two_level(d["x"].cuda())
        wq, ws, wts = bs.q4_quantize_two_level(w.cuda())
        y = bs.gemm_fp4(xq, xs, wq, ws, K, out_dtype=torch.bfloat16, a_tensor_scale=xts, b_tensor_scale=wts)
    torch.cuda.synchronize()
    assert bs.device_status()[0] == 0
    oa, osa, ta = oracle.q4_quantize_two_level(d["x"])
    ob, osb, tb = oracle.q4_quantize_two_level(w)
    assert np.array_equal(xq.cpu().numpy(), oa) and np.array_equal(wq.cpu().numpy(), ob)
    yr, s = oracle.gemm_fp4(oa, osa, ob, osb, K, alpha=ta * tb)
    yg = y.float().cpu().numpy()
    ok, ratio, rel = gemm_errors(yg, yr, s, True)
    tok, tratio = tight_errors(yg, yr, s, True)
    assert ok and tok, (ratio, rel, tratio)


def test_two_level_scale_not_with_lowrank(cuda_lib):
    bs = cuda_lib
    d = workloads.dense_lowrank(M=128, N=128, K=256)
    xq, xs, lt = bs.q4_quantize(d["x"].cuda(), lora_a_t=d["lora_a"].t().contiguous().cuda())
    wq, ws, wts = bs.q4_quantize_two_level(d["w"].cuda())
    with pytest.raises(bs.BSError) as e:
        bs.gemm_fp4(xq, xs, wq, ws, 256, lora_t=lt, lora_b_t=d["lora_b"].t().contiguous().cuda(), b_tensor_scale=wts)
    assert e.value.status == bs.BS_ERR_UNSUPPORTED


# ---------------------------------------------------------------------------
# W8A8: FP8 with one scale per token row of X and per channel (row) of W
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,K,dtype", [(1, 4096, torch.bfloat16), (130, 256, torch.float32),
                                       (7168, 4096, torch.bfloat16), (5, 128, torch.bfloat16)])
def test_q8_row_bit_exact(cuda_lib, M, K, dtype):
    bs = cuda_lib
    if M == 7168:
        x = workloads.fp8_sweep(1)["w"]
    else:
        g = torch.Generator().manual_seed(M + K)
        x = torch.randn(M, K, generator=g)
        x[:, 3] *= 50
        if M > 2:
            x[2] = 0
        x = x.to(dtype)
    codes, scales = bs.q8_quantize(x.cuda(), mode=bs.Q8_ROW)
    torch.cuda.synchronize()
    oc, os_ = oracle.q8_quantize_rowwise(x)
    assert np.array_equal(scales.cpu().numpy(), os_)
    assert np.array_equal(codes.cpu().numpy(), oc)


SCHEDULES = {"stream_k": 1, "per_tile": 2}


@pytest.mark.parametrize("schedule", sorted(SCHEDULES))
@pytest.mark.parametrize("M,N,K,rows", [(1, 7168, 4096, None), (16, 7168, 4096, None), (128, 7168, 4096, None),
                                        (4096, 7168, 4096, [0, 1, 127, 128, 2047, 4000, 4095]),
                                        (3, 256, 256, None), (100, 384, 512, None), (17, 640, 1024, None)])
def test_gemm_fp8_w8a8(cuda_lib, schedule, M, N, K, rows):
    """Y = s_x[m] s_w[n] sum_k a b against the oracle, bf16 output."""
    bs = cuda_lib
    if N == 7168:
        d = workloads.fp8_sweep(M)
        x, w = d["x"], d["w"]
    else:
        g = torch.Generator().manual_seed(M + N + K)
        x = torch.randn(M, K, generator=g).to(torch.bfloat16)
        w = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    with bs.kernel_options(fp8_stream_k=SCHEDULES[schedule]):
        xq, xs = bs.q8_quantize(x.cuda(), mode=bs.Q8_ROW)
        wq, ws = bs.q8_quantize(w.cuda(), mode=bs.Q8_ROW)
        y = bs.gemm_fp8(xq, xs, wq, ws, rowwise=True)
        y2 = bs.gemm_fp8(xq, xs, wq, ws, rowwise=True, weights_ready=True)
    torch.cuda.synchronize()
    assert bs.device_status()[0] == 0
    assert torch.equal(y, y2)
    rows = np.arange(M) if rows is None else np.asarray(rows)
    oa, osa = oracle.q8_quantize_rowwise(x[rows])
    ob, osb = oracle.q8_quantize_rowwise(w)
    assert np.array_equal(xq.cpu().numpy()[rows], oa)
    yr, s = oracle.gemm_fp8_rowwise(oa, osa, ob, osb)
    yg = y.float().cpu().numpy()[rows]
    ok, ratio, rel = gemm_errors(yg, yr, s, True)
    tok, tratio = tight_errors(yg, yr, s, True)
    assert ok and tok, (ratio, rel, tratio)
