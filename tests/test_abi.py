"""The C-ABI library loads, exports every symbol include/bsgemm.h declares, and
rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bsgemm.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import fp8_quantized_gemm_q4_gb300 as bs
    return bs.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "return")))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("q4_quantize", "q8_quantize", "bs_gemm", "bs_gemm_multi", "bs_grouped_gemm", "bs_grouped_gemm_swiglu_q4",
              "bs_moe_dispatch",
              "bs_moe_finalize", "bs_moe_combine", "bs_sf_bytes", "bs_sf_offset", "bs_get_device_status"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_sf_layout_helpers(lib):
    import fp8_quantized_gemm_q4_gb300 as bs
    assert bs.sf_bytes(128, 64) == 512
    assert bs.sf_bytes(1, 64) == 512          # rows pad to 128
    assert bs.sf_bytes(129, 128) == 2 * 128 * 8
    # tile (rb, kc) = rb * (K/64) + kc; inside: (r % 32) * 16 + (r / 32) * 4 + j
    K = 256
    assert bs.sf_offset(0, 0, K) == 0
    assert bs.sf_offset(0, 3, K) == 3
    assert bs.sf_offset(0, 4, K) == 512
    assert bs.sf_offset(1, 0, K) == 16
    assert bs.sf_offset(32, 0, K) == 4
    assert bs.sf_offset(127, 15, K) == 3 * 512 + 31 * 16 + 3 * 4 + 3
    assert bs.sf_offset(128, 0, K) == 4 * 512
    # the map is a bijection onto [0, sf_bytes)
    rows = 256
    offs = {bs.sf_offset(r, g, K) for r in range(rows) for g in range(K // 16)}
    assert offs == set(range(bs.sf_bytes(rows, K)))


def test_host_validation_rejects_before_launch(lib):
    import fp8_quantized_gemm_q4_gb300 as bs
    P = ctypes.c_void_p
    fake = P(1 << 20)        # never dereferenced: validation fails first
    # K not a multiple of 64
    assert lib.q4_quantize(fake, 1, 4, 100, 100, None, fake, fake, None, 0, None, None) == bs.BS_ERR_ALIGN
    # null output
    assert lib.q4_quantize(fake, 1, 4, 64, 64, None, None, fake, None, 0, None, None) == bs.BS_ERR_INVALID
    # bad dtype
    assert lib.q4_quantize(fake, 7, 4, 64, 64, None, fake, fake, None, 0, None, None) == bs.BS_ERR_INVALID
    # misaligned input pointer
    assert lib.q4_quantize(P((1 << 20) + 2), 1, 4, 64, 64, None, fake, fake, None, 0, None, None) == bs.BS_ERR_ALIGN
    # low-rank with the wrong rank
    assert lib.q4_quantize(fake, 1, 4, 64, 64, None, fake, fake, fake, 16, fake, None) == bs.BS_ERR_INVALID
    # M == 0 is a no-op
    assert lib.q4_quantize(None, 1, 0, 64, 64, None, None, None, None, 0, None, None) == bs.BS_OK
    # q8: K % 128
    assert lib.q8_quantize(fake, 1, 4, 64, 64, 1, fake, fake, None) == bs.BS_ERR_ALIGN
    assert lib.q8_quantize(fake, 1, 4, 128, 128, 7, fake, fake, None) == bs.BS_ERR_INVALID   # no such mode
    # two-level FP4: K % 64, null amax / tensor scale; tensor amax: K % 8
    assert lib.q4_quantize_two_level(fake, 1, 4, 96, 96, fake, fake, fake, fake, None) == bs.BS_ERR_ALIGN
    assert lib.q4_quantize_two_level(fake, 1, 4, 64, 64, None, fake, fake, fake, None) == bs.BS_ERR_INVALID
    assert lib.bs_tensor_amax(fake, 1, 4, 12, 12, fake, None) == bs.BS_ERR_ALIGN
    # router: k outside [1, min(E, 32)], E outside [1, 1024]
    assert lib.bs_moe_router_topk(fake, 4, 8, 9, fake, fake, None) == bs.BS_ERR_INVALID
    assert lib.bs_moe_router_topk(fake, 4, 2048, 8, fake, fake, None) == bs.BS_ERR_INVALID
    assert lib.bs_moe_router_topk(None, 0, 64, 8, None, None, None) == bs.BS_OK
    g = bs.GemmArgs()
    g.fmt, g.a, g.sfa, g.b, g.sfb, g.out = 0, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20
    g.M, g.N, g.K, g.alpha, g.ldo, g.out_dtype = 64, 100, 128, 1.0, 128, 1
    assert lib.bs_gemm(ctypes.byref(g), None) == bs.BS_ERR_ALIGN      # N % 128
    g.N = 128
    g.out = None
    assert lib.bs_gemm(ctypes.byref(g), None) == bs.BS_ERR_INVALID    # null out
    g.out = 1 << 20
    g.ldo = 100
    assert lib.bs_gemm(ctypes.byref(g), None) == bs.BS_ERR_ALIGN      # ldo
    g.ldo = 128
    # per-call kernel choices out of range, and a negative wait limit
    for field, bad in (("fp4_kernel", 3), ("fp4_stage_k", 64), ("fp4_small_experts", -1), ("fp4_half_tail", 5),
                       ("fp8_stream_k", 9), ("wait_timeout_us", -1), ("weights_ready", 2), ("fp8_scaling", 3)):
        setattr(g, field, bad)
        assert lib.bs_gemm(ctypes.byref(g), None) == bs.BS_ERR_INVALID, field
        assert field.encode() in lib.bs_last_error()
        setattr(g, field, 0)
    g.fmt = 9
    assert lib.bs_gemm(ctypes.byref(g), None) in (bs.BS_ERR_INVALID, bs.BS_ERR_CUDA)
    g.fmt = 0
    # grouped: E out of range, bad epilogue
    assert lib.bs_grouped_gemm(ctypes.byref(g), 0, fake, fake, 0, None, None, None, 0, None) == bs.BS_ERR_INVALID
    assert lib.bs_grouped_gemm(ctypes.byref(g), 4, fake, fake, 7, None, None, None, 0, None) == bs.BS_ERR_INVALID
    # COMBINE without routing tables
    assert lib.bs_grouped_gemm(ctypes.byref(g), 4, fake, fake, 2, None, None, None, 0, None) == bs.BS_ERR_INVALID
    # dispatch: workspace too small / bad E
    assert lib.bs_moe_dispatch(fake, fake, 8, 2, 2, fake, fake, fake, fake, fake, fake, 1, None) == bs.BS_ERR_INVALID
    assert lib.bs_moe_dispatch(fake, fake, 8, 2, 0, fake, fake, fake, fake, fake, fake, 1 << 20, None) == bs.BS_ERR_INVALID
    assert lib.bs_moe_rows_bound(8, 2, 2) == 16 + 2 * 127
    assert lib.bs_moe_finalize(P((1 << 20) + 4), fake, 8, None) == bs.BS_ERR_ALIGN
    # ROWS needs fp32 output and weight_of (g.out_dtype is bf16 here)
    assert lib.bs_grouped_gemm(ctypes.byref(g), 4, fake, fake, 3, None, fake, None, 0, None) == bs.BS_ERR_INVALID
    # gate/up GEMM with h quantized in the epilogue: out must be NULL (h goes
    # to h_codes / h_sf), both present and 16-byte aligned, E in range
    q4 = lib.bs_grouped_gemm_swiglu_q4
    assert q4(ctypes.byref(g), 4, fake, fake, fake, fake, None) == bs.BS_ERR_INVALID   # g.out is set
    g.out = None
    assert q4(ctypes.byref(g), 4, fake, fake, None, fake, None) == bs.BS_ERR_INVALID
    assert q4(ctypes.byref(g), 4, fake, fake, fake, P((1 << 20) + 4), None) == bs.BS_ERR_ALIGN
    assert q4(ctypes.byref(g), 0, fake, fake, fake, fake, None) == bs.BS_ERR_INVALID
    assert q4(ctypes.byref(g), 4, None, fake, fake, fake, None) == bs.BS_ERR_INVALID
    g.out = 1 << 20
    # combine: bad k, H not a multiple of 8, misaligned rows; T = 0 is a no-op
    assert lib.bs_moe_combine(fake, 64, fake, 128, 4, 0, 64, fake, fake, 64, None) == bs.BS_ERR_INVALID
    assert lib.bs_moe_combine(fake, 64, fake, 128, 4, 2, 60, fake, fake, 64, None) == bs.BS_ERR_ALIGN
    assert lib.bs_moe_combine(P((1 << 20) + 4), 64, fake, 128, 4, 2, 64, fake, fake, 64, None) == bs.BS_ERR_ALIGN
    assert lib.bs_moe_combine(None, 64, None, 0, 0, 2, 64, None, None, 64, None) == bs.BS_OK
    # multi-weight FP8: G out of range, null arrays, FP4, W8A8, M > 32, a null or
    # misaligned product operand -- all rejected before any device query
    arr3 = (P * 3)(fake, fake, fake)
    bad = (P * 3)(fake, None, fake)
    mis = (P * 3)(fake, P((1 << 20) + 8), fake)
    g.fmt, g.M, g.N, g.K, g.ldo = 1, 16, 128, 256, 128
    multi = lib.bs_gemm_multi
    assert multi(ctypes.byref(g), 0, arr3, arr3, arr3, None) == bs.BS_ERR_INVALID
    assert multi(ctypes.byref(g), 9, arr3, arr3, arr3, None) == bs.BS_ERR_INVALID
    assert multi(ctypes.byref(g), 3, None, arr3, arr3, None) == bs.BS_ERR_INVALID
    assert multi(ctypes.byref(g), 3, bad, arr3, arr3, None) == bs.BS_ERR_INVALID
    assert multi(ctypes.byref(g), 3, arr3, arr3, mis, None) == bs.BS_ERR_ALIGN
    g.K = 192
    assert multi(ctypes.byref(g), 3, arr3, arr3, arr3, None) == bs.BS_ERR_ALIGN     # K % 128
    g.K = 256
    g.M = 33
    assert multi(ctypes.byref(g), 3, arr3, arr3, arr3, None) == bs.BS_ERR_UNSUPPORTED
    g.M = 16
    g.fp8_scaling = 2
    assert multi(ctypes.byref(g), 3, arr3, arr3, arr3, None) == bs.BS_ERR_UNSUPPORTED
    g.fp8_scaling = 0
    g.fmt = 5
    assert multi(ctypes.byref(g), 3, arr3, arr3, arr3, None) == bs.BS_ERR_INVALID
    g.fmt, g.K = 0, 320                                                              # FP4: K % 256
    assert multi(ctypes.byref(g), 3, arr3, arr3, arr3, None) == bs.BS_ERR_ALIGN
    g.K, g.col_scale = 256, 1 << 20                                                  # FP4: per-column scale
    assert multi(ctypes.byref(g), 3, arr3, arr3, arr3, None) == bs.BS_ERR_UNSUPPORTED
    g.col_scale, g.fp4_decode = None, 2                                              # FP4: decode kernel only
    assert multi(ctypes.byref(g), 3, arr3, arr3, arr3, None) == bs.BS_ERR_UNSUPPORTED
    g.fp4_decode = 0
    g.fmt, g.M = 1, 0
    assert multi(ctypes.byref(g), 3, arr3, arr3, arr3, None) == bs.BS_OK           # M == 0: nothing to do
    assert lib.bs_gemm_multi_workspace_bytes(ctypes.byref(g), 3) == 0
    g.fmt, g.M, g.N, g.K, g.ldo = 0, 64, 128, 128, 128
    assert lib.bs_status_string(5) == b"device pipeline wait timed out"
    assert b"K=100" in lib.bs_last_error() or lib.bs_last_error() != b""


def test_product_path_has_no_oracle_or_cpu_fallback():
    pkg = os.path.join(ROOT, "fp8_quantized_gemm_q4_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".hpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "liboracle" not in src, f


def test_multi_binding_checks_its_lists():
    """The binding's list checks for bs_gemm_multi (before any library call)."""
    import torch
    import fp8_quantized_gemm_q4_gb300 as bs
    a = torch.zeros(16, 256, dtype=torch.uint8)
    with pytest.raises(ValueError):
        bs.gemm_fp8_multi(a, torch.zeros(2, 16), [])
    with pytest.raises(ValueError):
        bs.gemm_fp4_multi(a[:, :128], torch.zeros(512, dtype=torch.uint8), [], 256)
    w = (torch.zeros(128, 256, dtype=torch.uint8), torch.zeros(1, 2))
    with pytest.raises(ValueError):
        bs.gemm_fp8_multi(a, torch.zeros(2, 16), [w, w], outs=[torch.zeros(16, 128)])
