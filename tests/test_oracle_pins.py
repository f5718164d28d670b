"""Pins of the FP64 oracle against facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: golden
values derived by hand from the pages (tests/golden/*, each cited), closed
forms, invariants, library routines (ml_dtypes / torch dtype casts, numpy
matmul) on cases where the method reduces to them, and brute force.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.conftest import read_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def test_e2m1_value_set():
    for code, val in read_golden("e2m1_values.txt"):
        got = oracle.e2m1_decode(int(code))
        assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))
    assert max(oracle.e2m1_table()) == 6.0 and len(set(oracle.e2m1_table())) == 15  # +-0 equal


def test_e2m1_round_nearest_even_and_saturation():
    for x, code, val in read_golden("e2m1_rne.txt"):
        c = oracle.e2m1_encode(float(x))
        assert c == int(code), (x, c, code)
        assert oracle.e2m1_decode(c) == float(val)


def test_e2m1_matches_ml_dtypes_sweep():
    ml = pytest.importorskip("ml_dtypes")
    g = np.random.default_rng(1)
    xs = np.concatenate([np.linspace(-7, 7, 5601, dtype=np.float32),
                         g.standard_normal(3000).astype(np.float32) * 3,
                         np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0],
                                  dtype=np.float32)])
    ref = xs.astype(ml.float4_e2m1fn).view(np.uint8) & 0xF
    got = np.array([oracle.e2m1_encode(float(v)) for v in xs], dtype=np.uint8)
    assert np.array_equal(ref, got)


def test_e2m1_signed_zero():
    """E2M1 carries a sign bit, so -0 is its own code (0b1000); a -0.0 input
    divided by a positive group scale is -0.0 (IEEE division), so its code
    is 0b1000 in a quantized group too, as the library cast gives."""
    ml = pytest.importorskip("ml_dtypes")
    assert oracle.e2m1_encode(-0.0) == 0b1000 and oracle.e2m1_encode(0.0) == 0
    assert int(np.array([-0.0], dtype=np.float32).astype(ml.float4_e2m1fn).view(np.uint8)[0]) & 0xF == 0b1000
    x = np.zeros((1, 16), dtype=np.float32)
    x[0, 0], x[0, 3], x[0, 5] = 3.0, -0.0, -1e-3   # -1e-3 / 0.5 rounds to -0 as well
    codes, sf = oracle.q4_quantize(torch.from_numpy(x))
    nib = lambda k: (int(codes[0, k // 2]) >> (4 * (k & 1))) & 0xF
    assert nib(0) == 0b0111 and nib(3) == 0b1000 and nib(5) == 0b1000 and nib(1) == 0  # 3.0 / 0.5 = 6


def test_e4m3_facts():
    for code, val in read_golden("e4m3_facts.txt"):
        got = oracle.e4m3_decode(int(code))
        assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))
    fin = oracle.e4m3_table()[:127]
    assert np.all(np.diff(fin) > 0) and fin[-1] == 448.0


def test_e4m3_matches_torch_cast():
    g = np.random.default_rng(2)
    mags = np.exp(g.uniform(np.log(2.0 ** -12), np.log(448.0), 20000)).astype(np.float32)
    xs = np.concatenate([mags, -mags, oracle.e4m3_table()[:127].astype(np.float32),
                         ((oracle.e4m3_table()[1:127] + oracle.e4m3_table()[:126]) / 2).astype(np.float32)])
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in xs], dtype=np.uint8)
    assert np.array_equal(ref, got)


def test_e4m3_saturates():
    # up to the largest finite doubles: every value at or above 448 is 448
    # (for magnitudes ~2^53 x 448 a distance-based search sees only ties)
    for v in (448.0, 449.0, 463.9, 464.0, 500.0, 1e6, 2.0 ** 62, 1e30, 3.3895313892515355e38, 1e300):
        assert oracle.e4m3_encode(v) == 0x7E
        assert oracle.e4m3_encode(-v) == 0xFE


def test_e2m1_saturates_at_any_magnitude():
    for v in (6.0, 7.0, 1e6, 2.0 ** 60, 1e30, 1e300):
        assert oracle.e2m1_encode(v) == 0x7
        assert oracle.e2m1_encode(-v) == 0xF


def test_q4_quantize_huge_groups_saturate():
    # amax / 6 far above 448: the scale saturates to 448 and the codes of the
    # group (x / 448, still far above 6) saturate to +-6
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, 0], x[0, 1], x[0, 16] = 3e38, -1e30, 1e20
    c, s = oracle.q4_quantize(x)
    assert list(s.ravel()) == [0x7E, 0x7E]
    assert c[0, 0] == (0x7 | (0xF << 4)) and c[0, 8] == 0x7


# ---------------------------------------------------------------------------
# quantizers
# ---------------------------------------------------------------------------

def _lib_q4(x):
    """FP4 group-16 quantization with library casts (ml_dtypes E2M1, torch e4m3)."""
    ml = pytest.importorskip("ml_dtypes")
    x = np.asarray(x, dtype=np.float32)
    M, K = x.shape
    grp = np.abs(x.reshape(M, K // 16, 16)).max(axis=2)
    # torch's e4m3 cast does not saturate (>= 464 gives NaN); the scale saturates at 448
    s_code = torch.from_numpy(np.minimum(grp / np.float32(6), np.float32(448)).astype(np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    s = torch.from_numpy(s_code).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    s_full = np.repeat(s, 16, axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (x / s_full).astype(np.float32)
    codes = q.astype(ml.float4_e2m1fn).view(np.uint8) & 0xF
    codes[s_full == 0] = 0
    return codes, s_code


def _quant_inputs(seed=3, M=24, K=128):
    g = np.random.default_rng(seed)
    x = g.standard_normal((M, K)).astype(np.float32)
    x[0, :16] = 0.0                                   # zero group -> s = 0 -> codes 0
    x[1, 16:32] *= np.float32(1e-4)                   # subnormal / zero e4m3 scale
    x[2, :] *= np.float32(2000.0)                     # amax/6 > 448 -> saturated scale
    x[3, 32:48] = np.float32(6.0) * np.float32(0.171875)  # exact grid points
    x[4, :] = -np.abs(x[4, :]) * np.float32(1e-3)
    if M > 5:
        x[5, :16] = np.linspace(-3, 3, 16, dtype=np.float32)
    return x


def test_q4_quantize_matches_library_casts():
    x = _quant_inputs()
    ref_codes, ref_sf = _lib_q4(x)
    codes, sf = oracle.q4_quantize(x)
    assert np.array_equal(sf, ref_sf)
    assert np.array_equal(oracle.unpack_e2m1(codes, x.shape[1]), ref_codes)


def test_q4_quantize_bf16_input_and_packing():
    xb = torch.from_numpy(_quant_inputs(seed=4, M=8, K=64)).to(torch.bfloat16)
    codes, sf = oracle.q4_quantize(xb)
    ref_codes, ref_sf = _lib_q4(xb.float().numpy())
    assert np.array_equal(sf, ref_sf)
    # packing: element 2i in the low nibble, 2i+1 in the high nibble
    assert np.array_equal(codes, (ref_codes[:, 0::2] | (ref_codes[:, 1::2] << 4)).astype(np.uint8))


def test_q4_brute_force_nearest_and_error_bound():
    """Each code is a nearest grid point of x/s (brute force over all 16 codes)."""
    x = _quant_inputs(seed=5, M=6, K=64)
    codes, sf = oracle.q4_quantize(x)
    c = oracle.unpack_e2m1(codes, 64)
    for m in range(6):
        for k in range(64):
            s = oracle.e4m3_decode(sf[m, k // 16])
            if s == 0:
                assert c[m, k] == 0
                continue
            q = np.float32(x[m, k]) / np.float32(s)
            dists = [abs(oracle.e2m1_decode(cc) - float(q)) for cc in range(16)]
            if abs(q) <= 6:
                assert abs(oracle.e2m1_decode(c[m, k]) - float(q)) == min(dists)
                # dequantization error at most half the local grid spacing times s
                assert abs(oracle.e2m1_decode(c[m, k]) * s - x[m, k]) <= 1.0 * s + 1e-30
            else:
                assert abs(oracle.e2m1_decode(c[m, k])) == 6.0


def test_q4_scale_is_nearest_e4m3_of_amax_over_6():
    x = _quant_inputs(seed=6, M=6, K=64)
    _, sf = oracle.q4_quantize(x)
    fin = oracle.e4m3_table()[:127]
    for m in range(6):
        for g in range(4):
            t = float(np.float32(np.abs(x[m, g * 16:(g + 1) * 16]).max()) / np.float32(6))
            d = np.abs(fin - t)
            assert d[sf[m, g]] == d.min()


def test_q8_quantize_matches_library_casts():
    g = np.random.default_rng(7)
    x = g.standard_normal((5, 256)).astype(np.float32)
    x[:, 7] *= 50
    x[2, 128:] = 0
    codes, scales = oracle.q8_quantize(x, rows_per_block=1)
    amax = np.abs(x.reshape(5, 2, 128)).max(axis=2)
    s = (amax / np.float32(448)).astype(np.float32)
    assert np.array_equal(scales, s)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (x / np.repeat(s, 128, axis=1)).astype(np.float32)
    q[np.repeat(s, 128, axis=1) == 0] = 0
    ref = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)


def test_q8_block_128x128_scales():
    g = np.random.default_rng(8)
    w = (g.standard_normal((256, 256)) * 0.02).astype(np.float32)
    w[130, 5] = 3.0
    codes, scales = oracle.q8_quantize(w, rows_per_block=128)
    assert scales.shape == (2, 2)
    assert scales[1, 0] == np.float32(3.0) / np.float32(448)
    for rb in range(2):
        for kb in range(2):
            blk = w[rb * 128:(rb + 1) * 128, kb * 128:(kb + 1) * 128]
            assert scales[rb, kb] == np.float32(np.abs(blk).max()) / np.float32(448)


# ---------------------------------------------------------------------------
# GEMMs
# ---------------------------------------------------------------------------

def _dequant_fp4_lib(codes, sf, K):
    ml = pytest.importorskip("ml_dtypes")
    c = oracle.unpack_e2m1(codes, K)
    vals = c.view(ml.float4_e2m1fn).astype(np.float64)
    s = torch.from_numpy(np.ascontiguousarray(sf)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return vals * np.repeat(s, 16, axis=1)


@pytest.mark.parametrize("K,expect,sfc", [tuple(r) for r in read_golden("fp4_gemm_allones.txt")])
def test_gemm_fp4_all_ones_closed_form(K, expect, sfc):
    K = int(K)
    a, sa = oracle.q4_quantize(np.ones((3, K), np.float32))
    b, sb = oracle.q4_quantize(np.ones((5, K), np.float32))
    assert np.all(sa == int(sfc)) and np.all(sb == int(sfc))
    y, s = oracle.gemm_fp4(a, sa, b, sb, K)
    assert np.all(y == float(expect)) and np.all(s == float(expect))


def test_gemm_fp4_identity_weights_return_dequantized_x():
    K = 64
    g = np.random.default_rng(9)
    x = g.standard_normal((4, K)).astype(np.float32)
    a, sa = oracle.q4_quantize(x)
    b, sb = oracle.q4_quantize(np.eye(K, dtype=np.float32))
    y, _ = oracle.gemm_fp4(a, sa, b, sb, K)
    xhat = _dequant_fp4_lib(a, sa, K)
    assert np.array_equal(y, xhat * 1.03125)   # identity rows dequantize to 1.03125


def test_gemm_fp4_matches_matmul_of_dequantized():
    g = np.random.default_rng(10)
    for (M, N, K) in [(1, 1, 16), (3, 4, 32), (4, 3, 48), (2, 5, 64)]:
        x = g.standard_normal((M, K)).astype(np.float32)
        w = g.standard_normal((N, K)).astype(np.float32)
        a, sa = oracle.q4_quantize(x)
        b, sb = oracle.q4_quantize(w)
        y, s = oracle.gemm_fp4(a, sa, b, sb, K)
        xa, wb = _dequant_fp4_lib(a, sa, K), _dequant_fp4_lib(b, sb, K)
        ref = xa @ wb.T
        assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
        assert np.allclose(s, np.abs(xa) @ np.abs(wb).T, rtol=1e-12, atol=1e-12)


def test_gemm_fp4_scale_linearity():
    g = np.random.default_rng(11)
    x = g.standard_normal((3, 64)).astype(np.float32)
    w = g.standard_normal((4, 64)).astype(np.float32)
    b, sb = oracle.q4_quantize(w)
    a0, sa0 = oracle.q4_quantize(x)
    y0, _ = oracle.gemm_fp4(a0, sa0, b, sb, 64)
    for j in (1, 3, -2):
        a1, sa1 = oracle.q4_quantize(x * np.float32(2.0 ** j))
        assert np.array_equal(a1, a0)
        assert np.array_equal(sa1.astype(int), sa0.astype(int) + 8 * j)  # exponent field + j
        y1, _ = oracle.gemm_fp4(a1, sa1, b, sb, 64)
        assert np.array_equal(y1, y0 * 2.0 ** j)


def test_gemm_fp4_lowrank_bias_alpha_colscale():
    g = np.random.default_rng(12)
    M, N, K, r = 3, 5, 32, 4
    x = g.standard_normal((M, K)).astype(np.float32)
    w = g.standard_normal((N, K)).astype(np.float32)
    A = (g.standard_normal((K, r)) * 0.02).astype(np.float32)
    B = (g.standard_normal((r, N)) * 0.02).astype(np.float32)
    bias = (g.standard_normal(N) * 0.1).astype(np.float32)
    cs = g.uniform(0.5, 2, N).astype(np.float32)
    a, sa = oracle.q4_quantize(x)
    b, sb = oracle.q4_quantize(w)
    t = oracle.lowrank_t(x, A)
    assert np.allclose(t, x.astype(np.float64) @ A.astype(np.float64), rtol=1e-13, atol=1e-15)
    y, s = oracle.gemm_fp4(a, sa, b, sb, K, alpha=0.75, col_scale=cs, t=t, lora_b=B, bias=bias)
    main = _dequant_fp4_lib(a, sa, K) @ _dequant_fp4_lib(b, sb, K).T
    ref = 0.75 * cs[None, :].astype(np.float64) * main + t @ B.astype(np.float64) + bias[None, :]
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_gemm_fp8_matches_matmul_of_dequantized():
    g = np.random.default_rng(13)
    M, N, K = 3, 256, 256
    x = g.standard_normal((M, K)).astype(np.float32)
    x[:, 3] *= 50
    w = (g.standard_normal((N, K)) * 0.02).astype(np.float32)
    a, sa = oracle.q8_quantize(x, 1)
    b, sb = oracle.q8_quantize(w, 128)
    y, s = oracle.gemm_fp8(a, sa, b, sb)
    dq = lambda c: torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    xa = dq(a) * np.repeat(sa.astype(np.float64), 128, axis=1)
    wb = dq(b) * np.repeat(np.repeat(sb.astype(np.float64), 128, axis=1), 128, axis=0)[:N]
    assert np.allclose(y, xa @ wb.T, rtol=1e-12, atol=1e-12)
    # the quantized product approximates the fp32 product (fp8: 3 mantissa bits)
    assert np.abs(y - x.astype(np.float64) @ w.T.astype(np.float64)).max() < 0.05 * s.max()


# ---------------------------------------------------------------------------
# MoE
# ---------------------------------------------------------------------------

def test_moe_dispatch_hand_case():
    gold = {r[0]: [int(v) for v in r[1:]] for r in read_golden("moe_dispatch_2x8.txt")}
    ids = np.array([[t % 2, 1 - t % 2] for t in range(8)], dtype=np.int32)
    counts, offsets, por = oracle.moe_dispatch(ids, E=2, block=128)
    assert counts.tolist() == gold["counts"]
    assert offsets.tolist() == gold["offsets"]
    assert por[0:8].tolist() == gold["expert0_pairs"]
    assert por[128:136].tolist() == gold["expert1_pairs"]
    assert np.all(por[8:128] == -1) and np.all(por[136:] == -1)


def test_moe_dispatch_properties():
    g = np.random.default_rng(14)
    T, k, E = 300, 4, 9
    # k distinct experts per token, expert 4 never chosen (an empty expert)
    ids = np.stack([g.choice([e for e in range(E) if e != 4], k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, por = oracle.moe_dispatch(ids, E=E, block=128)
    assert counts[4] == 0 and offsets[5] == offsets[4]
    assert np.array_equal(counts, np.bincount(ids.ravel(), minlength=E))
    assert np.all(offsets % 128 == 0)
    real = por[por >= 0]
    assert sorted(real.tolist()) == list(range(T * k))
    for e in range(E):
        seg = por[offsets[e]:offsets[e] + counts[e]]
        assert np.all(ids.ravel()[seg] == e) and np.all(np.diff(seg) > 0)
        assert np.all(por[offsets[e] + counts[e]:offsets[e + 1]] == -1)


def test_swiglu_closed_forms():
    g = np.array([0.0, 50.0, -50.0, 1.0, -1.0])
    u = np.array([3.0, 2.0, 2.0, 1.0, 1.0])
    h = oracle.swiglu(g, u)
    assert h[0] == 0.0 and abs(h[1] - 100.0) < 1e-12 and abs(h[2]) < 1e-18
    assert abs(h[3] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    assert abs(h[3] - h[4] - 1.0) < 1e-15   # silu(x) - silu(-x) = x


def _quantized_experts(weights):
    gu = [oracle.q4_quantize(wgu) for wgu, _ in weights]
    dn = [oracle.q4_quantize(wd) for _, wd in weights]
    return [c for c, _ in gu], [s for _, s in gu], [c for c, _ in dn], [s for _, s in dn]


def test_moe_layer_all_ones_hand_case():
    gold = {r[0]: float(r[1]) for r in read_golden("moe_layer_allones.txt")}
    H = F = 32
    weights = [(np.full((2 * F, H), v, np.float32), np.full((H, F), v, np.float32)) for v in (1.0, 2.0)]
    x = np.ones((3, H), np.float32)
    ids = np.array([[0, 1]] * 3, dtype=np.int32)
    w = np.full((3, 2), 0.5, np.float32)
    res = oracle.moe_layer(x, ids, w, *_quantized_experts(weights), F=F)
    assert np.all(res["out"] == gold["out"])
    assert np.all(res["inter"][0]["h"] == gold["h_expert0"])
    assert np.all(res["inter"][1]["h"] == gold["h_expert1"])
    assert np.all(res["inter"][0]["y"] == gold["y_expert0"])
    assert np.all(res["inter"][1]["y"] == gold["y_expert1"])


def test_moe_layer_expert_relabel_invariance():
    g = np.random.default_rng(15)
    T, H, F, E, k = 4, 32, 16, 3, 2
    x = g.standard_normal((T, H)).astype(np.float32)
    weights = [((g.standard_normal((2 * F, H)) * 0.3).astype(np.float32),
                (g.standard_normal((H, F)) * 0.3).astype(np.float32)) for _ in range(E)]
    ids = np.array([[0, 1], [2, 0], [1, 2], [0, 2]], dtype=np.int32)
    w = g.uniform(0.1, 1, (T, k)).astype(np.float32)
    base = oracle.moe_layer(x, ids, w, *_quantized_experts(weights), F=F)["out"]
    perm = np.array([2, 0, 1])             # new label of old expert e is perm[e]
    inv = np.argsort(perm)
    relab = oracle.moe_layer(x, perm[ids], w, *_quantized_experts([weights[i] for i in inv]), F=F)["out"]
    assert np.array_equal(base, relab)
    # swapping the two slots of each token (with their weights) also changes nothing
    swapped = oracle.moe_layer(x, ids[:, ::-1], w[:, ::-1], *_quantized_experts(weights), F=F)["out"]
    assert np.allclose(base, swapped, rtol=2 ** -8, atol=0)


def test_moe_layer_top1_single_expert_is_dense_ffn():
    g = np.random.default_rng(16)
    T, H, F = 3, 32, 16
    x = g.standard_normal((T, H)).astype(np.float32)
    wgu = (g.standard_normal((2 * F, H)) * 0.3).astype(np.float32)
    wd = (g.standard_normal((H, F)) * 0.3).astype(np.float32)
    res = oracle.moe_layer(x, np.zeros((T, 1), np.int32), np.ones((T, 1), np.float32),
                           *_quantized_experts([(wgu, wd)]), F=F)
    # dense path written with library pieces: dequantize + numpy matmul + silu
    a, sa = oracle.q4_quantize(x)
    gw, gs = oracle.q4_quantize(wgu)
    gu = _dequant_fp4_lib(a, sa, H) @ _dequant_fp4_lib(gw, gs, H).T
    gg, uu = gu[:, :F], gu[:, F:]
    h = torch.from_numpy(gg / (1 + np.exp(-gg)) * uu).to(torch.bfloat16).float().numpy()
    hq, hs = oracle.q4_quantize(h)
    dw, ds = oracle.q4_quantize(wd)
    y = _dequant_fp4_lib(hq, hs, F) @ _dequant_fp4_lib(dw, ds, F).T
    ref = torch.from_numpy(y).to(torch.bfloat16).double().numpy()
    assert np.array_equal(res["out"], ref)


def _quantized_experts_fp8(weights):
    """Expert weights in FP8 e4m3 with 128x128 block scales (oracle quantizer)."""
    gu = [oracle.q8_quantize(wgu, 128) for wgu, _ in weights]
    dn = [oracle.q8_quantize(wd, 128) for _, wd in weights]
    return [c for c, _ in gu], [s for _, s in gu], [c for c, _ in dn], [s for _, s in dn]


def test_moe_layer_fp8_all_ones_hand_case():
    gold = {r[0]: float(r[1]) for r in read_golden("moe_layer_fp8_allones.txt")}
    H = F = 128
    weights = [(np.full((2 * F, H), v, np.float32), np.full((H, F), v, np.float32)) for v in (1.0, 2.0)]
    x = np.ones((2, H), np.float32)
    ids = np.array([[0, 1]] * 2, dtype=np.int32)
    w = np.full((2, 2), 0.5, np.float32)
    res = oracle.moe_layer(x, ids, w, *_quantized_experts_fp8(weights), F=F, fmt="fp8")
    assert np.all(res["out"] == gold["out"])
    for e in (0, 1):
        it = res["inter"][e]
        assert np.all(it["g"] == gold[f"g_expert{e}"]) and np.all(it["u"] == gold[f"g_expert{e}"])
        assert np.all(it["h"] == gold[f"h_expert{e}"])
        assert np.all(it["y"] == gold[f"y_expert{e}"])


def test_moe_layer_fp8_top1_single_expert_is_dense_ffn():
    """The FP8 layer with one expert and weight 1 is the dense FFN written with
    library pieces: torch's e4m3 cast to dequantize, numpy matmul, silu."""
    g = np.random.default_rng(17)
    T, H, F = 3, 256, 128
    x = g.standard_normal((T, H)).astype(np.float32)
    x[:, 5] *= 40
    wgu = (g.standard_normal((2 * F, H)) * 0.05).astype(np.float32)
    wd = (g.standard_normal((H, F)) * 0.05).astype(np.float32)
    res = oracle.moe_layer(x, np.zeros((T, 1), np.int32), np.ones((T, 1), np.float32),
                           *_quantized_experts_fp8([(wgu, wd)]), F=F, fmt="fp8")
    dq = lambda c: torch.from_numpy(np.ascontiguousarray(c)).view(torch.float8_e4m3fn).to(torch.float64).numpy()

    def tok(v):            # per 1x128 token block
        c, s_ = oracle.q8_quantize(v, 1)
        return dq(c) * np.repeat(s_.astype(np.float64), 128, axis=1)

    def blk(v):            # per 128x128 weight block
        c, s_ = oracle.q8_quantize(v, 128)
        return dq(c) * np.repeat(np.repeat(s_.astype(np.float64), 128, axis=1), 128, axis=0)[:v.shape[0]]

    gu = tok(x) @ blk(wgu).T
    gg, uu = gu[:, :F], gu[:, F:]
    for t in range(T):
        assert np.allclose(res["inter"][t]["g"], gg[t], rtol=1e-12, atol=1e-12)
        assert np.allclose(res["inter"][t]["u"], uu[t], rtol=1e-12, atol=1e-12)
    h = torch.from_numpy(gg / (1 + np.exp(-gg)) * uu).to(torch.bfloat16).float().numpy()
    y = tok(h) @ blk(wd).T
    for t in range(T):
        assert np.array_equal(res["inter"][t]["h"], h[t].astype(np.float64))
        assert np.allclose(res["inter"][t]["y"], y[t], rtol=1e-12, atol=1e-12)
    ref = torch.from_numpy(y).to(torch.bfloat16).double().numpy()
    assert np.array_equal(res["out"], ref)


def test_moe_layer_fp8_expert_relabel_invariance():
    g = np.random.default_rng(18)
    T, H, F, E, k = 4, 128, 128, 3, 2
    x = g.standard_normal((T, H)).astype(np.float32)
    weights = [((g.standard_normal((2 * F, H)) * 0.3).astype(np.float32),
                (g.standard_normal((H, F)) * 0.3).astype(np.float32)) for _ in range(E)]
    ids = np.array([[0, 1], [2, 0], [1, 2], [0, 2]], dtype=np.int32)
    w = g.uniform(0.1, 1, (T, k)).astype(np.float32)
    base = oracle.moe_layer(x, ids, w, *_quantized_experts_fp8(weights), F=F, fmt="fp8")["out"]
    perm = np.array([1, 2, 0])
    inv = np.argsort(perm)
    relab = oracle.moe_layer(x, perm[ids], w, *_quantized_experts_fp8([weights[i] for i in inv]), F=F,
                             fmt="fp8")["out"]
    assert np.array_equal(base, relab)
    # the FP8 layer differs from the FP4 one on the same weights (the format is used)
    fp4 = oracle.moe_layer(x, ids, w, *_quantized_experts(weights), F=F)["out"]
    assert not np.array_equal(base, fp4)


# ---------------------------------------------------------------------------
# top-k router ("DeepGEMM for Hopper MoE", section 1) and bf16 rounding
# ---------------------------------------------------------------------------

def test_moe_router_hand_case():
    rows = {r[0]: r[1:] for r in read_golden("moe_router_hand.txt")}
    for t in range(3):
        lg = np.array([[float(v) for v in rows[f"logits{t}"]]], dtype=np.float32)
        ids, w = oracle.moe_router(lg, 3)
        assert ids[0].tolist() == [int(v) for v in rows[f"ids{t}"]]
        assert np.allclose(w[0], [float(v) for v in rows[f"w{t}"]], rtol=1e-14, atol=0)


def test_moe_router_matches_numpy_brute_force():
    """numpy's stable sort of -logits (ties keep the lower index first) and a
    float64 softmax of the chosen logits, on logits rounded to one decimal so
    that ties are frequent."""
    g = np.random.default_rng(7)
    for E, k in ((8, 2), (64, 8), (256, 8), (13, 13)):
        lg = np.round(g.standard_normal((200, E)), 1).astype(np.float32)
        ids, w = oracle.moe_router(lg, k)
        ref = np.argsort(-lg, axis=1, kind="stable")[:, :k]
        assert np.array_equal(ids, ref)
        ch = np.take_along_axis(lg.astype(np.float64), ref, axis=1)
        ex = np.exp(ch - ch.max(axis=1, keepdims=True))
        assert np.allclose(w, ex / ex.sum(axis=1, keepdims=True), rtol=1e-13, atol=0)


def test_moe_router_invariants():
    g = np.random.default_rng(8)
    # multiples of 2^-10 below 2^12 in magnitude: adding 4 below is exact in fp32
    lg = (np.round(g.standard_normal((50, 32)) * 3 * 1024) / 1024).astype(np.float32)
    ids, w = oracle.moe_router(lg, 8)
    assert np.allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert np.all(np.diff(w, axis=1) <= 0)                 # descending logit -> descending weight
    ids2, w2 = oracle.moe_router(lg + np.float32(4.0), 8)   # a shift of every logit changes nothing
    assert np.array_equal(ids, ids2) and np.allclose(w, w2, rtol=1e-12)
    ids3, w3 = oracle.moe_router(lg, 32)                    # k = E: the full softmax over all experts
    full = np.exp(lg.astype(np.float64) - lg.max(axis=1, keepdims=True))
    full /= full.sum(axis=1, keepdims=True)
    assert np.allclose(np.take_along_axis(full, ids3, axis=1), w3, rtol=1e-13)


def test_round_bf16_single_rounding():
    import torch
    # fp32-representable values: torch's fp32 -> bf16 cast is one rounding
    g = np.random.default_rng(9)
    v = np.concatenate([g.standard_normal(4000) * 10.0 ** g.integers(-30, 30, 4000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.01171875, -2.5, 3.0e38]]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_bf16(v.astype(np.float64)), ref)
    # a value just above a bf16 midpoint that fp32 rounds onto the midpoint:
    # rounding twice (fp64 -> fp32 -> bf16) would go down to 1, once goes up
    assert oracle.round_bf16([1 + 2.0 ** -8 + 2.0 ** -30])[0] == 1 + 2.0 ** -7
    assert oracle.round_bf16([1 + 2.0 ** -8])[0] == 1.0                    # tie to even
    assert oracle.round_bf16([1 + 3 * 2.0 ** -8])[0] == 1 + 2.0 ** -6      # tie to even (up)
    assert oracle.round_bf16([1e-40])[0] == 2.0 ** -133                    # bf16 subnormal spacing
    assert np.isinf(oracle.round_bf16([3.4e38])[0])


# ---------------------------------------------------------------------------
# format variants: two-level FP4, W8A8 per-row FP8 ("Tencent AI Infra
# interview notes": scale-granularity table, W8A8 SmoothQuant)
# ---------------------------------------------------------------------------

def test_q4_two_level_exponent_is_the_smallest_that_fits():
    assert oracle.q4_two_level_exp(0.0) == 0
    for amax in (2688.0, 2688.0001, 1344.0, 1344.0001, 0.1, 0.02, 3.0e-30, 1.0e30, 6.0, 448.0 * 6 * 2 ** -20):
        e = oracle.q4_two_level_exp(amax)
        a = float(np.float32(amax))
        assert a <= 6 * 448 * 2.0 ** e          # the largest group scale does not exceed 448
        assert a > 6 * 448 * 2.0 ** (e - 1)     # and one power of two less would


def test_q4_two_level_is_one_level_on_the_scaled_tensor():
    """Codes and group scales equal the library casts' quantization of the
    tensor divided (exactly) by its power-of-two scale."""
    g = np.random.default_rng(11)
    for std in (0.02, 1.0, 300.0):
        x = (g.standard_normal((6, 128)) * std).astype(np.float32)
        x[1, 16:32] = 0
        codes, sf, ts = oracle.q4_quantize_two_level(x)
        e = oracle.q4_two_level_exp(np.abs(x).max())
        assert ts == 2.0 ** e
        ref_codes, ref_sf = _lib_q4(np.ldexp(x, -e).astype(np.float32))
        assert np.array_equal(sf, ref_sf)
        assert np.array_equal(oracle.unpack_e2m1(codes, 128), ref_codes)


def test_q4_two_level_scales_use_the_top_binade_and_dequantize():
    g = np.random.default_rng(12)
    x = (g.standard_normal((16, 256)) * 0.02).astype(np.float32)
    codes, sf, ts = oracle.q4_quantize_two_level(x)
    smax = oracle.e4m3_decode(int(sf.max()))
    assert 256.0 <= smax <= 448.0
    c = oracle.unpack_e2m1(codes, 256)
    s = np.vectorize(oracle.e4m3_decode)(sf).repeat(16, axis=1)
    deq = np.vectorize(oracle.e2m1_decode)(c) * s * ts
    assert np.all(np.abs(deq - x) <= s * ts + 1e-30)     # within one unit of the local grid
    # the point of the second level: N(0, 0.02) weights, whose one-level group
    # scales are e4m3 subnormals with 2-3 significant bits, lose less (over
    # 256 groups the mean error drops by about 6 %)
    c1, sf1 = oracle.q4_quantize(x)
    s1 = np.vectorize(oracle.e4m3_decode)(sf1).repeat(16, axis=1)
    deq1 = np.vectorize(oracle.e2m1_decode)(oracle.unpack_e2m1(c1, 256)) * s1
    assert np.abs(deq - x).mean() < 0.97 * np.abs(deq1 - x).mean()


def test_q8_rowwise_matches_library_casts():
    g = np.random.default_rng(13)
    x = g.standard_normal((5, 384)).astype(np.float32)
    x[:, 7] *= 50
    x[3, :] = 0
    codes, scales = oracle.q8_quantize_rowwise(x)
    s = (np.abs(x).max(axis=1) / np.float32(448)).astype(np.float32)
    assert np.array_equal(scales, s)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (x / s[:, None]).astype(np.float32)
    q[s == 0] = 0
    ref = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)


def test_gemm_fp8_rowwise_matches_matmul_of_dequantized():
    g = np.random.default_rng(14)
    xa = g.standard_normal((9, 256)).astype(np.float32)
    xb = (g.standard_normal((130, 256)) * 0.02).astype(np.float32)
    a, sa = oracle.q8_quantize_rowwise(xa)
    b, sb = oracle.q8_quantize_rowwise(xb)
    y, s = oracle.gemm_fp8_rowwise(a, sa, b, sb)
    da = torch.from_numpy(a).view(torch.float8_e4m3fn).to(torch.float64).numpy() * sa[:, None]
    db = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy() * sb[:, None]
    ref = da @ db.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    assert np.all(s >= np.abs(y) - 1e-12)
