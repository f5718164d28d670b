"""Dense block-scaled FP4 GEMM on the GPU vs the FP64 oracle.

Tolerance: |y - y_ref| <= 1e-3 * S + 2^-8 |y_ref| (bf16 output only),
S = sum_k |a_k b_k| (+ low-rank and bias magnitudes).  A tighter diagnostic
bound (1e-4 S) is asserted too, so a dropped K group cannot hide in the slack.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.helpers import gemm_errors, tight_errors

pytestmark = pytest.mark.gpu

# The library runs FP4 GEMMs on CTA pairs (256 x 256 tiles) by default; the
# one-CTA kernel (128 x 256) and the 128-deep K stages are per-call choices
# (bs_gemm_args.fp4_kernel / fp4_stage_k).  Every case runs on each variant.
VARIANTS = {"pair": (2, 256), "one_cta": (1, 256), "pair_bk128": (2, 128), "one_cta_bk128": (1, 128)}


@pytest.fixture(autouse=True, params=sorted(VARIANTS))
def fp4_variant(request):
    kernel, bk = VARIANTS[request.param]
    import fp8_quantized_gemm_q4_gb300 as bs
    with bs.kernel_options(fp4_kernel=kernel, fp4_stage_k=bk):
        yield request.param


def run_case(bs, x, w, out_dtype, alpha=1.0, col_scale=None, lora=None, bias=None, rows=None):
    K = x.shape[1]
    xq, xs, lt = bs.q4_quantize(x.cuda(), lora_a_t=None if lora is None else lora[0].t().contiguous().cuda())
    wq, ws, _ = bs.q4_quantize(w.cuda())
    y = bs.gemm_fp4(xq, xs, wq, ws, K, out_dtype=out_dtype, alpha=alpha,
                    col_scale=None if col_scale is None else col_scale.cuda(),
                    lora_t=lt, lora_b_t=None if lora is None else lora[1].t().contiguous().cuda(),
                    bias=None if bias is None else bias.cuda())
    torch.cuda.synchronize()
    assert bs.device_status()[0] == 0
    rows = np.arange(x.shape[0]) if rows is None else np.asarray(rows)
    oa, osa = oracle.q4_quantize(x[rows])
    ob, osb = oracle.q4_quantize(w)
    assert np.array_equal(xq.cpu().numpy()[rows], oa)
    t = None if lora is None else oracle.lowrank_t(x[rows], lora[0])
    yr, s = oracle.gemm_fp4(oa, osa, ob, osb, K, alpha=alpha, col_scale=col_scale, t=t,
                            lora_b=None if lora is None else lora[1], bias=bias)
    yg = y.float().cpu().numpy()[rows]
    bf = out_dtype == torch.bfloat16
    ok, ratio, rel = gemm_errors(yg, yr, s, bf)
    tok, tratio = tight_errors(yg, yr, s, bf)
    return ok, ratio, rel, tok, tratio


def test_dense_tiny_fp32(cuda_lib):
    """Workload 0: X[128,512] W[256,512] fp32 N(0,1), fp32 output."""
    d = workloads.dense_tiny()
    ok, ratio, rel, tok, tratio = run_case(cuda_lib, d["x"], d["w"], torch.float32)
    assert ok and tok, (ratio, rel, tratio)


@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (100, 384, 192), (300, 256, 320), (129, 640, 1024),
                                   (512, 1024, 2048)])
def test_ragged_shapes(cuda_lib, M, N, K):
    g = torch.Generator().manual_seed(M + N + K)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    w = torch.randn(N, K, generator=g).to(torch.bfloat16)
    for dt in (torch.float32, torch.bfloat16):
        ok, ratio, rel, tok, tratio = run_case(cuda_lib, x, w, dt)
        assert ok and tok, (dt, ratio, rel, tratio)


def test_alpha_colscale_bias(cuda_lib):
    g = torch.Generator().manual_seed(5)
    M, N, K = 257, 512, 1024
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    w = torch.randn(N, K, generator=g).to(torch.bfloat16)
    cs = torch.rand(N, generator=g) + 0.5
    b = (torch.randn(N, generator=g) * 0.1).to(torch.bfloat16)
    ok, ratio, rel, tok, tratio = run_case(cuda_lib, x, w, torch.bfloat16, alpha=0.5, col_scale=cs, bias=b)
    assert ok and tok, (ratio, rel, tratio)


def test_small_weights_subnormal_scales(cuda_lib):
    """N(0, 0.02) weights give e4m3 scales in the subnormal range."""
    g = torch.Generator().manual_seed(6)
    x = torch.randn(256, 512, generator=g).to(torch.bfloat16)
    w = (torch.randn(256, 512, generator=g) * 0.02).to(torch.bfloat16)
    _, ws = oracle.q4_quantize(w)
    assert (ws < 8).mean() > 0.5     # most scales are e4m3 subnormals (exponent field 0)
    ok, ratio, rel, tok, tratio = run_case(cuda_lib, x, w, torch.float32)
    assert ok and tok, (ratio, rel, tratio)


def test_lowrank_and_bias(cuda_lib):
    d = workloads.dense_lowrank(M=200, N=384, K=512)
    ok, ratio, rel, tok, tratio = run_case(cuda_lib, d["x"], d["w"], torch.bfloat16,
                                           lora=(d["lora_a"], d["lora_b"]), bias=d["bias"])
    assert ok and tok, (ratio, rel, tratio)


def test_full_size_lowrank_sampled_rows(cuda_lib, fp4_variant):
    """Workload 1 at full size (8192^3, low-rank branch, bias, bf16 out), checked on
    rows spanning the first, middle and last tiles."""
    if fp4_variant.endswith("bk128"):
        pytest.skip("full size runs on the 256-deep variants")
    d = workloads.dense_lowrank()
    rows = [0, 1, 31, 32, 127, 128, 4095, 4096, 8000, 8191]
    ok, ratio, rel, tok, tratio = run_case(cuda_lib, d["x"], d["w"], torch.bfloat16,
                                           lora=(d["lora_a"], d["lora_b"]), bias=d["bias"], rows=rows)
    assert ok and tok, (ratio, rel, tratio)


@pytest.mark.parametrize("half_tail", [1, 2])
def test_short_last_wave_half_tiles(cuda_lib, half_tail):
    """80 pair tiles (2560 x 2048) on at most 76 pairs: the last 4 tiles run as
    eight 256 x 128 half tiles on CTA pairs (fp4_half_tail = 1, the default;
    2 keeps whole tiles)."""
    d = workloads.dense_lowrank(M=2560, N=2048, K=256)
    with cuda_lib.kernel_options(fp4_half_tail=half_tail):
        for kw in ({}, {"lora": (d["lora_a"], d["lora_b"]), "bias": d["bias"]}):
            for dt in (torch.bfloat16, torch.float32):
                if kw and dt == torch.float32:
                    continue
                ok, ratio, rel, tok, tratio = run_case(cuda_lib, d["x"], d["w"], dt, **kw)
                assert ok and tok, (dt, bool(kw), ratio, rel, tratio)


def test_empty_m_is_noop(cuda_lib):
    bs = cuda_lib
    a = torch.empty((0, 32), dtype=torch.uint8, device="cuda")
    sfa = torch.empty(16, dtype=torch.uint8, device="cuda")
    b = torch.zeros((128, 32), dtype=torch.uint8, device="cuda")
    sfb = torch.zeros(bs.sf_bytes(128, 64), dtype=torch.uint8, device="cuda")
    y = bs.gemm_fp4(a, sfa, b, sfb, 64)
    assert y.shape == (0, 128)


def test_unsupported_lowrank_with_alpha(cuda_lib):
    bs = cuda_lib
    d = workloads.dense_lowrank(M=128, N=128, K=256)
    xq, xs, lt = bs.q4_quantize(d["x"].cuda(), lora_a_t=d["lora_a"].t().contiguous().cuda())
    wq, ws, _ = bs.q4_quantize(d["w"].cuda())
    with pytest.raises(bs.BSError) as e:
        bs.gemm_fp4(xq, xs, wq, ws, 256, alpha=2.0, lora_t=lt, lora_b_t=d["lora_b"].t().contiguous().cuda())
    assert e.value.status == bs.BS_ERR_UNSUPPORTED
