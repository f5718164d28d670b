"""The pins must catch plausible mistakes in the oracle.

Each case compiles a copy of oracle.c with one planted mistake (on the CPU)
and runs the pin suite against it in a subprocess; the suite must fail.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "wrong_fp4_max": ("div_f32(amax, 6.0f)", "div_f32(amax, 4.0f)"),
    "dropped_b_scale": ("double sb = orc_e4m3_decode(j->sfb[n * G + g]);", "double sb = 1.0;"),
    "wrong_group_index": ("double sa = orc_e4m3_decode(j->sfa[m * G + g]);",
                          "double sa = orc_e4m3_decode(j->sfa[m * G]);"),
    "swapped_nibbles": ("e2m1_at(j->b, j->K / 2, n, k)", "e2m1_at(j->b, j->K / 2, n, k ^ 1)"),
    "ties_to_odd": ("(c & 1) == 0 && (best & 1) == 1", "(c & 1) == 1 && (best & 1) == 0"),
    "fp8_block_index": ("j->sb8[(n / 128) * KB + kb]", "j->sb8[(n % 2) * KB + kb]"),
    "fp8_no_scale_rounding": ("float s = div_f32(amax, 448.0f);", "float s = (float)(amax / 447.0);"),
    "dispatch_unaligned": ("int32_t padded = (counts[e] + block - 1) / block * block;",
                           "int32_t padded = counts[e];"),
    "lowrank_sign": ("y += prod;\n                    s += fabs(prod);", "y -= prod;\n                    s += fabs(prod);"),
    "swiglu_sign": ("h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];", "h[i] = g[i] / (1.0 + exp(g[i])) * u[i];"),
    "negative_zero_code": ("return signbit(v) ? (uint8_t)(c | 8) : c;", "return (v < 0) ? (uint8_t)(c | 8) : c;"),
    "e4m3_subnormal_scale": ("? ldexp((double)m / 8.0, -6)", "? ldexp((double)m / 8.0, -7)"),
    "scale_not_rounded": ("float s = (float)orc_e4m3_decode(sc);", "float s = div_f32(amax, 6.0f);"),
    "dispatch_reversed": ("for (int64_t p = 0; p < T * k; ++p)\n            if (topk_ids[p] == e)",
                          "for (int64_t p = T * k - 1; p >= 0; --p)\n            if (topk_ids[p] == e)"),
    "bias_dropped": ("if (j->bias) { y += j->bias[n]; s += fabs(j->bias[n]); }",
                     "if (j->bias) { s += fabs(j->bias[n]); }"),
    "fp8_token_scale_index": ("double sa = j->sa8[m * KB + kb];", "double sa = j->sa8[m * KB];"),
    "fp8_block_amax_one_row": ("for (int64_t m = r0; m < r1; ++m)\n                for (int j = 0; j < 128; ++j) {\n"
                               "                    float a = fabsf",
                               "for (int64_t m = r0; m < r0 + 1; ++m)\n                for (int j = 0; j < 128; ++j) {\n"
                               "                    float a = fabsf"),
    "ties_away_from_zero": ("(d == best_d && (c & 1) == 0 && (best & 1) == 1)", "(d == best_d && c > best)"),
    "router_ties_to_higher_id": ("if (best < 0 || l[e] > l[best]) best = e;", "if (best < 0 || l[e] >= l[best]) best = e;"),
    "router_ascending": ("if (best < 0 || l[e] > l[best]) best = e;", "if (best < 0 || l[e] < l[best]) best = e;"),
    "router_softmax_over_all_experts": ("for (int j = 0; j < k; ++j) sum += exp((double)l[ids[t * k + j]] - top);",
                                        "for (int e = 0; e < E; ++e) sum += exp((double)l[e] - top);"),
    "bf16_truncates": ("const double r = rint(ldexp(a, -q))", "const double r = trunc(ldexp(a, -q))"),
    "bf16_nine_bits": ("int q = e - 8;", "int q = e - 9;"),
    "two_level_fits_448_not_6x448": ("while ((double)amax <= 2688.0 * ldexp(1.0, e - 1)) --e;",
                                     "while ((double)amax <= 448.0 * ldexp(1.0, e - 1)) --e;"),
    "two_level_scale_off_by_one": ("*tensor_scale = (float)ldexp(1.0, e);", "*tensor_scale = (float)ldexp(1.0, e + 1);"),
    "two_level_unscaled_input": ("xs[m * K + k] = (float)ldexp((double)x[m * ldx + k], -e);",
                                 "xs[m * K + k] = x[m * ldx + k];"),
    "rowwise_scale_447": ("const float srow = div_f32(amax, 448.0f);", "const float srow = div_f32(amax, 447.0f);"),
    "rowwise_gemm_drops_weight_scale": ("const double f = (double)sa[m] * (double)sb[n];",
                                        "const double f = (double)sa[m];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    assert src.count(old) == 1, name
    mutant = tmp_path / "oracle_mutant.c"
    mutant.write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so),
                           str(mutant), "-lm"])
    env = dict(os.environ, ORACLE_SO=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"


# Mistakes planted in the Python half of the oracle (the MoE layer's order of
# steps): the pin suite runs from a scratch tree whose `oracle` package is
# the mutated copy (the C library is the unchanged one, via ORACLE_SO).
PY_MUTANTS = {
    "gate_up_swapped": ("g, u = gu[0, :F], gu[0, F:]", "u, g = gu[0, :F], gu[0, F:]"),
    "h_not_rounded": ("h = round_bf16(swiglu(g, u))", "h = swiglu(g, u)"),
    "routing_weight_dropped": ("acc += w[t, slot] * y[0]", "acc += y[0]"),
    "output_not_rounded": ("out[i] = round_bf16(acc)", "out[i] = acc"),
    "fp8_layer_with_fp4_quantizer": ("quantize = q8_quantize", "quantize = q4_quantize"),
}


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_pins_catch_planted_mistake_in_layer(name, tmp_path):
    import oracle as real_oracle
    old, new = PY_MUTANTS[name]
    src = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    assert src.count(old) == 1, name
    pkg = tmp_path / "oracle"
    pkg.mkdir()
    (pkg / "__init__.py").write_text(src.replace(old, new))
    for d in ("tests", "workloads"):
        os.symlink(os.path.join(ROOT, d), tmp_path / d)
    env = dict(os.environ, ORACLE_SO=real_oracle.build())
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join("tests", "test_oracle_pins.py")],
                       cwd=str(tmp_path), env=env, capture_output=True, text=True, timeout=600)
    # a pin must fail on an assertion (not the tree failing to import)
    assert "ERROR" not in r.stdout and " failed" in r.stdout, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
