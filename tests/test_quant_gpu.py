"""GPU quantizers vs the FP64 oracle: codes and scales bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.helpers import sf_rowmajor

pytestmark = pytest.mark.gpu


def special_rows(x):
    """Plant edge cases: zero group, tiny (subnormal / zero scale), huge (saturated
    scale), exact grid points, negative values rounding to -0, ties."""
    x = x.clone()
    M, K = x.shape
    if M > 0:
        x[0, :16] = 0
    if M > 1:
        x[1, :] *= 1e-4
    if M > 2:
        x[2, :] *= 3000.0
    if M > 3:
        x[3, :16] = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * 2) * 0.171875 * (6.0 / 6.0)
    if M > 4:
        x[4, :] = -x[4, :].abs() * 1e-3
    if M > 5:
        x[5, 16:32] = 1e-12
    return x


@pytest.mark.parametrize("M,K,dtype", [(1, 64, torch.float32), (3, 128, torch.float32),
                                       (128, 512, torch.float32), (300, 320, torch.float32),
                                       (257, 1024, torch.bfloat16), (64, 8192, torch.bfloat16)])
def test_q4_quantize_bit_exact(cuda_lib, M, K, dtype):
    bs = cuda_lib
    g = torch.Generator().manual_seed(M * 7 + K)
    x = special_rows(torch.randn(M, K, generator=g)).to(dtype)
    codes, sf, _ = bs.q4_quantize(x.cuda())
    torch.cuda.synchronize()
    oc, os_ = oracle.q4_quantize(x)
    assert np.array_equal(codes.cpu().numpy(), oc)
    sfn = sf.cpu().numpy()
    assert np.array_equal(sf_rowmajor(sfn, M, K), os_)
    # padding rows of the last 128-row block carry zero scales
    Mpad = (M + 127) // 128 * 128
    if Mpad > M:
        pad = sf_rowmajor(sfn, Mpad, K)[M:]
        assert np.all(pad == 0)


def test_q4_quantize_gather(cuda_lib):
    bs = cuda_lib
    x = torch.randn(50, 256).to(torch.bfloat16)
    gather = torch.tensor([3, -1, 49, 0, 3, 17, -1, 8], dtype=torch.int32)
    codes, sf, _ = bs.q4_quantize(x.cuda(), gather=gather.cuda())
    rows = torch.stack([x[i] if i >= 0 else torch.zeros(256, dtype=x.dtype) for i in gather.tolist()])
    oc, os_ = oracle.q4_quantize(rows)
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(sf_rowmajor(sf.cpu().numpy(), 8, 256), os_)


def _all_bf16_under_every_scale():
    """Groups whose amax is 6 s for each finite positive e4m3 value s (so the
    group scale is exactly s), filled with every bf16 value of magnitude in
    (s / 8, 6 s] with both signs: every quotient x / s that can decide a code."""
    e4 = oracle.e4m3_table()[1:127]
    allbf = torch.arange(0, 1 << 15, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float()
    allbf = allbf[torch.isfinite(allbf) & (allbf > 0)]
    rows = []
    for sv in e4:
        sv = float(sv)
        vals = allbf[(allbf > sv / 8) & (allbf <= 6 * sv)]
        vals = torch.cat([vals, -vals])
        n = (len(vals) + 14) // 15 * 15
        vals = torch.cat([vals, torch.zeros(n - len(vals))]).view(-1, 15)
        head = torch.full((vals.shape[0], 1), 6 * sv)
        rows.append(torch.cat([head, vals], dim=1))
    g = torch.cat(rows).reshape(-1)
    pad = (-len(g)) % 256
    return torch.cat([g, torch.zeros(pad)]).view(-1, 256)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_q4_quantize_exhaustive_bf16_quotients(cuda_lib, dtype):
    bs = cuda_lib
    x = _all_bf16_under_every_scale().to(dtype)
    codes, sf, _ = bs.q4_quantize(x.cuda())
    torch.cuda.synchronize()
    oc, os_ = oracle.q4_quantize(x)
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(sf_rowmajor(sf.cpu().numpy(), x.shape[0], 256), os_)


def test_q4_lowrank_fused_exhaustive_bf16_quotients(cuda_lib):
    """The fused quantize + low-rank pass on the same exhaustive value set."""
    bs = cuda_lib
    x = _all_bf16_under_every_scale().to(torch.bfloat16)
    x = x.reshape(-1, 1024) if x.numel() % 1024 == 0 else torch.cat(
        [x.reshape(-1), torch.zeros((-x.numel()) % 1024, dtype=x.dtype)]).view(-1, 1024)
    a = (torch.randn(1024, 32) * 0.02).to(torch.bfloat16)
    codes, sf, _ = bs.q4_quantize(x.cuda(), lora_a_t=a.t().contiguous().cuda())
    torch.cuda.synchronize()
    oc, os_ = oracle.q4_quantize(x)
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(sf_rowmajor(sf.cpu().numpy(), x.shape[0], 1024), os_)


def _every_bf16_amax(K):
    """One 16-element group per finite positive bf16 value v: the group holds v
    (its amax), -v/2 and 0.7 v (rounded to bf16, both below v in magnitude), so
    the group scale e4m3(RN(v / 6)) is taken for every amax a bf16 input can
    have.  Rows of K elements, zero groups as padding."""
    allbf = torch.arange(1, 0x7F80, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float()
    g = torch.zeros(allbf.numel(), 16)
    g[:, 0] = allbf
    g[:, 5] = -allbf / 2
    g[:, 9] = allbf * 0.7
    per_row = K // 16
    pad = (-g.shape[0]) % per_row
    g = torch.cat([g, torch.zeros(pad, 16)])
    return g.reshape(-1, K).to(torch.bfloat16)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_q4_quantize_every_bf16_amax(cuda_lib, dtype):
    bs = cuda_lib
    x = _every_bf16_amax(256).to(dtype)
    codes, sf, _ = bs.q4_quantize(x.cuda())
    torch.cuda.synchronize()
    oc, os_ = oracle.q4_quantize(x)
    assert np.array_equal(sf_rowmajor(sf.cpu().numpy(), x.shape[0], 256), os_)
    assert np.array_equal(codes.cpu().numpy(), oc)


def test_q4_lowrank_fused_every_bf16_amax(cuda_lib):
    bs = cuda_lib
    x = _every_bf16_amax(1024)
    a = (torch.randn(1024, 32) * 0.02).to(torch.bfloat16)
    codes, sf, _ = bs.q4_quantize(x.cuda(), lora_a_t=a.t().contiguous().cuda())
    torch.cuda.synchronize()
    oc, os_ = oracle.q4_quantize(x)
    assert np.array_equal(sf_rowmajor(sf.cpu().numpy(), x.shape[0], 1024), os_)
    assert np.array_equal(codes.cpu().numpy(), oc)


@pytest.mark.parametrize("rows_in,rows_out,K", [(50, 8, 256), (4096, 1000, 4096), (7, 300, 64)])
def test_fp4_gather_rows_equals_quantize_with_gather(cuda_lib, rows_in, rows_out, K):
    bs = cuda_lib
    g = torch.Generator().manual_seed(rows_in + rows_out)
    x = special_rows(torch.randn(rows_in, K, generator=g)).to(torch.bfloat16).cuda()
    idx = torch.randint(-1, rows_in, (rows_out,), generator=g, dtype=torch.int32).cuda()
    c, s, _ = bs.q4_quantize(x)
    gc, gs = bs.fp4_gather_rows(c, s, K, idx)
    rc, rs, _ = bs.q4_quantize(x, gather=idx)
    torch.cuda.synchronize()
    assert torch.equal(gc, rc) and torch.equal(gs, rs)


def test_q4_quantize_full_size_activation(cuda_lib):
    """The 8192 x 8192 bf16 activation of the dense low-rank workload, every row."""
    bs = cuda_lib
    x = workloads.dense_lowrank(lowrank=False, bias=False)["x"]
    codes, sf, _ = bs.q4_quantize(x.cuda())
    torch.cuda.synchronize()
    rows = np.r_[0:64, 4000:4064, 8128:8192]
    oc, os_ = oracle.q4_quantize(x[rows])
    assert np.array_equal(codes.cpu().numpy()[rows], oc)
    assert np.array_equal(sf_rowmajor(sf.cpu().numpy(), 8192, 8192)[rows], os_)


@pytest.mark.parametrize("M,K", [(200, 1024), (130, 320), (64, 8192), (1000, 512), (20000, 256)])
def test_q4_lowrank_left_factor(cuda_lib, M, K):
    """Codes, scales and T = X A from one call (fused pass when K % 256 == 0,
    separate kernels otherwise), including row counts that leave the last
    32-row CTA of the fused pass partly empty."""
    bs = cuda_lib
    d = workloads.dense_lowrank(M=M, N=256, K=K)
    x, a = d["x"], d["lora_a"]
    codes, sf, lt = bs.q4_quantize(x.cuda(), lora_a_t=a.t().contiguous().cuda())
    torch.cuda.synchronize()
    oc, os_ = oracle.q4_quantize(x)
    assert np.array_equal(codes.cpu().numpy(), oc)
    sfn = sf.cpu().numpy()
    assert np.array_equal(sf_rowmajor(sfn, M, K), os_)
    Mpad = (M + 127) // 128 * 128
    assert np.all(sf_rowmajor(sfn, Mpad, K)[M:] == 0)
    t = lt.float().cpu().numpy().astype(np.float64)
    t_gpu = t[:, :32] + t[:, 32:]
    t_ref = oracle.lowrank_t(x, a)
    mag = np.abs(x.float().numpy().astype(np.float64)) @ np.abs(a.float().numpy().astype(np.float64))
    assert np.all(np.abs(t_gpu - t_ref) <= 1e-5 * mag + 2.0 ** -16 * np.abs(t_ref))
    assert np.all(t[:, 32:] == (t_gpu - t[:, :32]))  # lo is the bf16 remainder


def test_q4_lowrank_gather(cuda_lib):
    bs = cuda_lib
    d = workloads.dense_lowrank(M=40, N=256, K=512)
    x, a = d["x"], d["lora_a"]
    gather = torch.tensor([5, -1, 39, 0, 5] * 30, dtype=torch.int32)
    codes, sf, lt = bs.q4_quantize(x.cuda(), gather=gather.cuda(), lora_a_t=a.t().contiguous().cuda())
    rows = torch.stack([x[i] if i >= 0 else torch.zeros(512, dtype=x.dtype) for i in gather.tolist()])
    oc, os_ = oracle.q4_quantize(rows)
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(sf_rowmajor(sf.cpu().numpy(), len(gather), 512), os_)
    t = lt.float().cpu().numpy().astype(np.float64)
    t_ref = oracle.lowrank_t(rows, a)
    assert np.allclose(t[:, :32] + t[:, 32:], t_ref, rtol=1e-4, atol=1e-4)


@pytest.mark.parametrize("M,K,dtype", [(1, 4096, torch.bfloat16), (16, 4096, torch.bfloat16),
                                       (130, 256, torch.float32), (4096, 4096, torch.bfloat16)])
def test_q8_token_bit_exact(cuda_lib, M, K, dtype):
    bs = cuda_lib
    if K == 4096:
        x = workloads.fp8_sweep(M)["x"]
    else:
        x = special_rows(torch.randn(M, K)).to(dtype)
    codes, scales = bs.q8_quantize(x.cuda(), mode=bs.Q8_TOKEN)
    torch.cuda.synchronize()
    rows = np.arange(M) if M <= 256 else np.r_[0:128, M - 128:M]
    oc, os_ = oracle.q8_quantize(x[rows], rows_per_block=1)
    assert np.array_equal(codes.cpu().numpy()[rows], oc)
    assert np.array_equal(scales.cpu().numpy().T[rows], os_)   # [K/128, M] layout


@pytest.mark.parametrize("N,K", [(200, 384), (7168, 4096)])
def test_q8_block_bit_exact(cuda_lib, N, K):
    bs = cuda_lib
    if N == 7168:
        w = workloads.fp8_sweep(1)["w"]
    else:
        w = (torch.randn(N, K) * 0.02).to(torch.bfloat16)
    codes, scales = bs.q8_quantize(w.cuda(), mode=bs.Q8_BLOCK)
    torch.cuda.synchronize()
    oc, os_ = oracle.q8_quantize(w, rows_per_block=128)
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(scales.cpu().numpy(), os_)


def _q8_quotient_sweep(dtype, n_scales=512, seed=3, lo_exp=-12):
    """1 x 128 blocks whose first element A is the block amax, so the block
    scale is s = fl32(A / 448), for a spread of A over the positive finite
    bf16 range; the other 127 elements take every bf16 value of magnitude in
    [A 2^-12, A] with both signs (fp32 input: as many random fp32 values in
    that range).  These are the quotients x / s that decide the e4m3 codes,
    under n_scales different scales; rows of 32 blocks."""
    allbf = torch.arange(1, 0x7F80, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float()
    A = allbf[::len(allbf) // n_scales][:n_scales]
    g = torch.Generator().manual_seed(seed)
    blocks = []
    for a in A.tolist():
        if dtype == torch.bfloat16:
            vals = allbf[(allbf >= a * 2.0 ** lo_exp) & (allbf <= a)]
        else:
            vals = a * torch.exp2(lo_exp * torch.rand(3000, generator=g))
        vals = torch.cat([vals, -vals])
        n = (len(vals) + 126) // 127 * 127
        vals = torch.cat([vals, torch.zeros(n - len(vals))]).view(-1, 127)
        blocks.append(torch.cat([torch.full((vals.shape[0], 1), a), vals], dim=1))
    b = torch.cat(blocks)
    b = torch.cat([b, torch.zeros((-b.shape[0]) % 32, 128)])
    return b.reshape(-1, 4096).to(dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_q8_token_quotient_sweep(cuda_lib, dtype):
    """FP8 1 x 128 codes and scales bit-exact against the oracle's correctly
    rounded division over every bf16 quotient under 512 block scales."""
    bs = cuda_lib
    x = _q8_quotient_sweep(dtype)
    codes, scales = bs.q8_quantize(x.cuda(), mode=bs.Q8_TOKEN)
    torch.cuda.synchronize()
    oc, os_ = oracle.q8_quantize(x, rows_per_block=1)
    assert np.array_equal(scales.cpu().numpy().T, os_)
    assert np.array_equal(codes.cpu().numpy(), oc)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_q8_token_small_quotient_sweep(cuda_lib, dtype):
    """The same sweep down to quotients of 448 * 2^-20 (below half the
    smallest e4m3 subnormal): every decision point of the e4m3 subnormal
    range, under 64 scales."""
    bs = cuda_lib
    x = _q8_quotient_sweep(dtype, n_scales=64, seed=4, lo_exp=-20)
    codes, scales = bs.q8_quantize(x.cuda(), mode=bs.Q8_TOKEN)
    torch.cuda.synchronize()
    oc, os_ = oracle.q8_quantize(x, rows_per_block=1)
    assert np.array_equal(scales.cpu().numpy().T, os_)
    assert np.array_equal(codes.cpu().numpy(), oc)


def _q8_midpoint_rows(n_scales=64, seed=5):
    """fp32 blocks [A, x ...] whose x make x / s land on and within three fp32
    ulps of every e4m3 decision point (midpoints between consecutive e4m3
    values up to 448, normal and subnormal), both signs, s = fl32(A / 448)
    for n_scales random A."""
    g = np.random.default_rng(seed)
    mags = np.unique(np.abs(oracle.e4m3_table()))
    mags = mags[np.isfinite(mags) & (mags <= 448)]
    mids = (mags[:-1] + mags[1:]) / 2
    blocks = []
    for _ in range(n_scales):
        a = np.float32(g.uniform(0.5, 4.0) * 2.0 ** int(g.integers(-8, 9)))
        sc = np.float32(np.float64(a) / 448.0)
        xs = []
        for m in mids:
            x0 = np.float32(m * np.float64(sc))
            up, dn = x0, x0
            xs.append(x0)
            for _ in range(3):
                up = np.nextafter(up, np.float32(np.inf), dtype=np.float32)
                dn = np.nextafter(dn, np.float32(0), dtype=np.float32)
                xs += [up, dn]
        xs = np.array([v for v in xs if 0 < v <= a], dtype=np.float32)
        xs = np.concatenate([xs, -xs])
        n = (len(xs) + 126) // 127 * 127
        xs = np.concatenate([xs, np.zeros(n - len(xs), np.float32)]).reshape(-1, 127)
        blocks.append(np.concatenate([np.full((xs.shape[0], 1), a, np.float32), xs], axis=1))
    b = np.concatenate(blocks)
    b = np.concatenate([b, np.zeros(((-b.shape[0]) % 32, 128), np.float32)])
    return torch.from_numpy(b.reshape(-1, 4096))


@pytest.mark.parametrize("mode", ["token", "row", "block"])
def test_q8_decision_points(cuda_lib, mode):
    """Quotients on and next to every e4m3 decision point (the cases the fast
    quotient hands to IEEE division), for the token, row and block modes."""
    bs = cuda_lib
    x = _q8_midpoint_rows()
    if mode == "token":
        codes, scales = bs.q8_quantize(x.cuda(), mode=bs.Q8_TOKEN)
        oc, os_ = oracle.q8_quantize(x, rows_per_block=1)
        os_ = os_.T
    elif mode == "block":
        codes, scales = bs.q8_quantize(x.cuda(), mode=bs.Q8_BLOCK)
        oc, os_ = oracle.q8_quantize(x, rows_per_block=128)
    else:
        codes, scales = bs.q8_quantize(x.cuda(), mode=bs.Q8_ROW)
        oc, os_ = oracle.q8_quantize_rowwise(x)
    torch.cuda.synchronize()
    assert np.array_equal(scales.cpu().numpy(), os_)
    assert np.array_equal(codes.cpu().numpy(), oc)


@pytest.mark.parametrize("K", [128, 384, 4096 + 128])
def test_q8_token_odd_block_counts(cuda_lib, K):
    """K % 256 == 128: the last 256-element unit of a row holds one block."""
    bs = cuda_lib
    x = special_rows(torch.randn(37, K)).to(torch.bfloat16)
    codes, scales = bs.q8_quantize(x.cuda(), mode=bs.Q8_TOKEN)
    torch.cuda.synchronize()
    oc, os_ = oracle.q8_quantize(x, rows_per_block=1)
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(scales.cpu().numpy().T, os_)
