"""FP64 CPU oracle for block-scaled FP4 / FP8 GEMM and the grouped MoE layer.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the product package.  The
arithmetic lives in ``oracle.c`` (plain C, double precision); this module
only compiles it with gcc, marshals numpy arrays and composes the MoE layer
from the C pieces in the pages' order.  Rounding of final results to bf16 /
fp32 is done here with torch's dtype casts (a library routine).

Pages cited (titles):
  * "Warp-specialised W4A4 kernel on the newest GPU architecture", section 1:
    Y = (Q(X) Q(W)^T) (.) scale + L(X) + b.
  * "Tencent AI Infra interview notes", FP4 format table and per-group
    quantized GEMM.
  * "DeepGEMM teardown (FP8 GEMM)", sections 2.1-2.3, 5.2, 5.3.
  * "DeepGEMM for Hopper MoE", sections 1 (gate -> top-k -> experts ->
    weighted sum), 2.1 (FP8 GEMM), 3.1 (fused swish).

Every function here has at least one pin in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

BLOCK_ROWS = 128  # MoE segment alignment (one MMA row tile)


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library with gcc (-O2, pthreads)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # ORACLE_SO lets the mutation test load a deliberately broken copy
            lib = ctypes.CDLL(os.environ.get("ORACLE_SO") or build())
            P, I64, D, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double, ctypes.c_int
            lib.orc_e2m1_decode.restype = D
            lib.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_decode.restype = D
            lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.orc_e2m1_encode.restype = ctypes.c_uint8
            lib.orc_e2m1_encode.argtypes = [D]
            lib.orc_e4m3_encode.restype = ctypes.c_uint8
            lib.orc_e4m3_encode.argtypes = [D]
            lib.orc_q4_quantize.argtypes = [P, I64, I64, I64, P, P]
            lib.orc_q8_quantize.argtypes = [P, I64, I64, I64, I, P, P]
            lib.orc_gemm_fp4.argtypes = [P, P, P, P, I64, I64, I64, D, P, P, P, I, P, P, P, I]
            lib.orc_gemm_fp8.argtypes = [P, P, P, P, I64, I64, I64, P, P, I]
            lib.orc_lowrank_t.argtypes = [P, I64, I64, I64, P, I, P]
            lib.orc_moe_rows_bound.restype = I64
            lib.orc_moe_rows_bound.argtypes = [I64, I, I, I]
            lib.orc_moe_dispatch.argtypes = [P, I64, I, I, I, P, P, P]
            lib.orc_swiglu.argtypes = [P, P, I64, P]
            lib.orc_moe_router.argtypes = [P, I64, I, I, P, P]
            lib.orc_round_bf16.restype = D
            lib.orc_round_bf16.argtypes = [D]
            lib.orc_q4_two_level_exp.restype = I
            lib.orc_q4_two_level_exp.argtypes = [ctypes.c_float]
            lib.orc_q4_quantize_two_level.argtypes = [P, I64, I64, I64, P, P, P]
            lib.orc_q8_quantize_rowwise.argtypes = [P, I64, I64, I64, P, P]
            lib.orc_gemm_fp8_rowwise.argtypes = [P, P, P, P, I64, I64, I64, P, P]
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(x):
    """Exact widening of bf16/fp16/fp32 input (numpy or torch) to fp32."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().to("cpu", torch.float32).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def e2m1_decode(code: int) -> float:
    return _load().orc_e2m1_decode(int(code) & 0xF)


def e4m3_decode(code: int) -> float:
    return _load().orc_e4m3_decode(int(code) & 0xFF)


def e2m1_encode(v: float) -> int:
    return int(_load().orc_e2m1_encode(float(v)))


def e4m3_encode(v: float) -> int:
    return int(_load().orc_e4m3_encode(float(v)))


E2M1_TABLE = None
E4M3_TABLE = None


def e2m1_table() -> np.ndarray:
    global E2M1_TABLE
    if E2M1_TABLE is None:
        E2M1_TABLE = np.array([e2m1_decode(c) for c in range(16)], dtype=np.float64)
    return E2M1_TABLE


def e4m3_table() -> np.ndarray:
    global E4M3_TABLE
    if E4M3_TABLE is None:
        E4M3_TABLE = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return E4M3_TABLE


def unpack_e2m1(codes: np.ndarray, K: int) -> np.ndarray:
    """Packed [R, K/2] bytes -> [R, K] 4-bit codes (low nibble = even k)."""
    codes = np.asarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape[:-1] + (K,), dtype=np.uint8)
    out[..., 0::2] = codes & 0xF
    out[..., 1::2] = codes >> 4
    return out


# ---------------------------------------------------------------------------
# quantizers
# ---------------------------------------------------------------------------

def q4_quantize(x):
    """FP4 E2M1 group-16 quantization.  Returns (codes u8 [M,K/2], sf u8 [M,K/16])."""
    x = _f32(x)
    M, K = x.shape
    assert K % 16 == 0
    codes = np.zeros((M, K // 2), dtype=np.uint8)
    sf = np.zeros((M, K // 16), dtype=np.uint8)
    if M:
        _load().orc_q4_quantize(_p(x), M, K, K, _p(codes), _p(sf))
    return codes, sf


def q8_quantize(x, rows_per_block: int = 1):
    """FP8 e4m3 quantization with fp32 scales per (rows_per_block x 128) block.

    Returns (codes u8 [M,K], scales f32 [ceil(M/rows_per_block), K/128])."""
    x = _f32(x)
    M, K = x.shape
    assert K % 128 == 0
    codes = np.zeros((M, K), dtype=np.uint8)
    nrb = (M + rows_per_block - 1) // rows_per_block
    scales = np.zeros((nrb, K // 128), dtype=np.float32)
    if M:
        _load().orc_q8_quantize(_p(x), M, K, K, int(rows_per_block), _p(codes), _p(scales))
    return codes, scales


def q4_two_level_exp(amax: float) -> int:
    """Exponent e of the two-level FP4 tensor scale 2^e: the smallest e with
    amax <= 6 * 448 * 2^e (0 for a zero tensor)."""
    return int(_load().orc_q4_two_level_exp(float(np.float32(amax))))


def q4_quantize_two_level(x):
    """Two-level FP4: a power-of-two tensor scale 2^e above the e4m3 group
    scales.  Returns (codes [M, K/2], group scales [M, K/16], tensor scale
    2^e as a float)."""
    x = _f32(x)
    M, K = x.shape
    codes = np.zeros((M, K // 2), dtype=np.uint8)
    sf = np.zeros((M, K // 16), dtype=np.uint8)
    ts = np.zeros(1, dtype=np.float32)
    _load().orc_q4_quantize_two_level(_p(x), M, K, K, _p(codes), _p(sf), _p(ts))
    return codes, sf, float(ts[0])


def q8_quantize_rowwise(x):
    """FP8 with one fp32 scale per row over all of K (W8A8: per-token
    activations, per-channel weights).  Returns (codes [M, K], scales [M])."""
    x = _f32(x)
    M, K = x.shape
    codes = np.zeros((M, K), dtype=np.uint8)
    scales = np.zeros(M, dtype=np.float32)
    if M:
        _load().orc_q8_quantize_rowwise(_p(x), M, K, K, _p(codes), _p(scales))
    return codes, scales


# ---------------------------------------------------------------------------
# GEMMs
# ---------------------------------------------------------------------------

def lowrank_t(x, a) -> np.ndarray:
    """T = X A in FP64 on the unquantized X (the left factor of L(X))."""
    x = _f32(x)
    a = _f32(a)
    M, K = x.shape
    r = a.shape[1]
    t = np.zeros((M, r), dtype=np.float64)
    if M:
        _load().orc_lowrank_t(_p(x), M, K, K, _p(a), r, _p(t))
    return t


def gemm_fp4(a_codes, sfa, b_codes, sfb, K, alpha=1.0, col_scale=None, t=None,
             lora_b=None, bias=None, nthreads=None):
    """FP64 block-scaled FP4 GEMM.  Returns (y [M,N] f64, s [M,N] f64) where s is
    the sum of |terms| used by the error bound."""
    a_codes = np.ascontiguousarray(a_codes, dtype=np.uint8)
    b_codes = np.ascontiguousarray(b_codes, dtype=np.uint8)
    sfa = np.ascontiguousarray(sfa, dtype=np.uint8)
    sfb = np.ascontiguousarray(sfb, dtype=np.uint8)
    M, N = a_codes.shape[0], b_codes.shape[0]
    cs = None if col_scale is None else np.ascontiguousarray(_f32(col_scale), dtype=np.float64)
    tt = None if t is None else np.ascontiguousarray(t, dtype=np.float64)
    lb = None if lora_b is None else np.ascontiguousarray(_f32(lora_b), dtype=np.float64)
    bb = None if bias is None else np.ascontiguousarray(_f32(bias), dtype=np.float64)
    r = 0 if tt is None else tt.shape[1]
    y = np.zeros((M, N), dtype=np.float64)
    s = np.zeros((M, N), dtype=np.float64)
    if M and N:
        _load().orc_gemm_fp4(_p(a_codes), _p(sfa), _p(b_codes), _p(sfb), M, N, K, float(alpha),
                             _p(cs), _p(tt), _p(lb), r, _p(bb), _p(y), _p(s),
                             nthreads or default_threads())
    return y, s


def gemm_fp8(a_codes, sa, b_codes, sb, nthreads=None):
    """FP64 FP8 GEMM with per (1x128) A scales and per (128x128) B scales."""
    a_codes = np.ascontiguousarray(a_codes, dtype=np.uint8)
    b_codes = np.ascontiguousarray(b_codes, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sb = np.ascontiguousarray(sb, dtype=np.float32)
    M, K = a_codes.shape
    N = b_codes.shape[0]
    y = np.zeros((M, N), dtype=np.float64)
    s = np.zeros((M, N), dtype=np.float64)
    if M and N:
        _load().orc_gemm_fp8(_p(a_codes), _p(sa), _p(b_codes), _p(sb), M, N, K, _p(y), _p(s),
                             nthreads or default_threads())
    return y, s


def gemm_fp8_rowwise(a_codes, sa, b_codes, sb):
    """W8A8 GEMM y = sa[m] sb[n] sum_k a b in FP64 (plus the error scale)."""
    a_codes = np.ascontiguousarray(a_codes, dtype=np.uint8)
    b_codes = np.ascontiguousarray(b_codes, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32).reshape(-1)
    sb = np.ascontiguousarray(sb, dtype=np.float32).reshape(-1)
    M, K = a_codes.shape
    N = b_codes.shape[0]
    y = np.zeros((M, N), dtype=np.float64)
    s = np.zeros((M, N), dtype=np.float64)
    if M and N:
        _load().orc_gemm_fp8_rowwise(_p(a_codes), _p(sa), _p(b_codes), _p(sb), M, N, K, _p(y), _p(s))
    return y, s


# ---------------------------------------------------------------------------
# MoE
# ---------------------------------------------------------------------------

def moe_dispatch(topk_ids, E: int, block: int = BLOCK_ROWS):
    """Contiguous, block-aligned per-expert grouping of (token, slot) pairs.

    Returns (counts [E], offsets [E+1], pair_of_row [offsets[E]])."""
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    T, k = ids.shape
    lib = _load()
    bound = lib.orc_moe_rows_bound(T, k, E, block)
    counts = np.zeros(E, dtype=np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    por = np.zeros(max(bound, 1), dtype=np.int32)
    lib.orc_moe_dispatch(_p(ids), T, k, E, block, _p(counts), _p(offsets), _p(por))
    return counts, offsets, por[: offsets[E]].copy()


def swiglu(g, u) -> np.ndarray:
    g = np.ascontiguousarray(g, dtype=np.float64)
    u = np.ascontiguousarray(u, dtype=np.float64)
    h = np.zeros_like(g)
    _load().orc_swiglu(_p(g), _p(u), g.size, _p(h))
    return h


def round_bf16(y) -> np.ndarray:
    """Round FP64 values to bf16 in one step (round to nearest, ties to even;
    orc_round_bf16) and return them as fp64."""
    y = np.asarray(y, dtype=np.float64)
    f = _load().orc_round_bf16
    return np.vectorize(f, otypes=[np.float64])(y) if y.size else y.copy()


def moe_router(logits, k: int):
    """Top-k routing of every token from its fp32 router logits ("DeepGEMM for
    Hopper MoE" section 1): expert ids int32 [T, k] in descending order of
    logit (ties to the lower id) and the softmax of the chosen logits, fp64
    [T, k]."""
    lg = _f32(logits)
    T, E = lg.shape
    assert 1 <= k <= E
    ids = np.zeros((T, k), dtype=np.int32)
    w = np.zeros((T, k), dtype=np.float64)
    if T:
        _load().orc_moe_router(_p(lg), T, E, k, _p(ids), _p(w))
    return ids, w


def moe_layer(x, topk_ids, topk_w, wgu_codes, wgu_sf, wd_codes, wd_sf, F: int,
              tokens=None, nthreads=None, fmt: str = "fp4"):
    """FP64 MoE layer ("DeepGEMM for Hopper MoE" section 1: experts then weighted
    sum; section 3.1 swish; "DeepGEMM teardown" 5.3 grouping), in the pages' order:

      1. group (token, slot) pairs by expert            (moe_dispatch)
      2. quantize each routed token's activations       (q4_quantize | q8_quantize)
      3. g = x^ Wg^T, u = x^ Wu^T per expert            (gemm_fp4 | gemm_fp8; Wg = rows [0,F), Wu = [F,2F))
      4. h = bf16(silu(g) * u)                          (swiglu + bf16 rounding)
      5. requantize h                                   (q4_quantize | q8_quantize)
      6. y = h^ Wd^T per expert                         (gemm_fp4 | gemm_fp8)
      7. out[t] = bf16(sum_slot w[t,slot] * y[t,slot])

    Formats: fmt "fp4" quantizes with q4_quantize and multiplies with gemm_fp4
    (E2M1 codes, e4m3 group-16 scales); fmt "fp8" quantizes x and h with
    q8_quantize per 1x128 token block and multiplies with gemm_fp8, the expert
    weights carrying 128x128 block scales ("DeepGEMM teardown" sections 2.2 and
    5.3; "DeepGEMM for Hopper MoE" section 2.1: FP8 grouped expert GEMMs).

    wgu_codes/wgu_sf: per-expert lists (or arrays) of the quantized [2F,H] gate/up
    weights; wd_codes/wd_sf: per-expert quantized [H,F] down weights.  Only the
    tokens in ``tokens`` (default: all) are evaluated; each output row depends on
    its own token only.  Returns dict with out (bf16-rounded f64 [len(tokens),H])
    and the per-pair intermediates keyed by pair index t*k+slot.
    """
    x = _f32(x)
    ids = np.asarray(topk_ids, dtype=np.int32)
    w = np.asarray(_f32(topk_w), dtype=np.float64)
    T, k = ids.shape
    H = x.shape[1]
    if tokens is None:
        tokens = np.arange(T)
    tokens = np.asarray(tokens)
    if fmt == "fp4":
        quantize = q4_quantize

        def gemm(a, sa, b, sb, K):
            return gemm_fp4(a, sa, b, sb, K, nthreads=nthreads)
    elif fmt == "fp8":
        quantize = q8_quantize

        def gemm(a, sa, b, sb, K):
            return gemm_fp8(a, sa, b, sb, nthreads=nthreads)
    else:
        raise ValueError(f"fmt must be 'fp4' or 'fp8', not {fmt!r}")
    out = np.zeros((len(tokens), H), dtype=np.float64)
    inter = {}
    for i, t in enumerate(tokens):
        xq, xs = quantize(x[t:t + 1])
        acc = np.zeros(H, dtype=np.float64)
        for slot in range(k):
            e = int(ids[t, slot])
            gu, gu_s = gemm(xq, xs, wgu_codes[e], wgu_sf[e], H)
            g, u = gu[0, :F], gu[0, F:]
            h = round_bf16(swiglu(g, u))
            hq, hs = quantize(h.astype(np.float32)[None, :])
            y, ys = gemm(hq, hs, wd_codes[e], wd_sf[e], F)
            acc += w[t, slot] * y[0]
            inter[int(t) * k + slot] = dict(g=g, u=u, h=h, y=y[0], s_gu=gu_s[0], s_y=ys[0])
        out[i] = round_bf16(acc)
    return dict(out=out, inter=inter)
