"""Block-scaled FP4 / FP8 GEMM for GB300 (sm_103a): Python binding.

Thin ctypes binding of the C ABI in ``include/bsgemm.h``: it marshals torch
tensors (device memory, the current stream) into the library's entry points
and allocates outputs with torch.  Every step of the computation runs in the
library's CUDA kernels; there is no fallback.  If ``libbsgemm.so`` has not
been built, ``load()`` raises.

    Y = (Q(X) Q(W)^T) (.) scale + L(X) + b
    ("Warp-specialised W4A4 kernel on the newest GPU architecture", section 1)
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from ._build import LIB as _LIB_PATH

__all__ = [
    "load", "sf_bytes", "sf_offset", "q4_quantize", "tensor_amax", "q4_quantize_two_level", "fp4_gather_rows", "fp8_gather_rows", "q8_quantize", "gemm_fp4", "gemm_fp8", "gemm_fp8_multi", "gemm_fp4_multi",
    "grouped_gemm_fp4", "grouped_gemm_fp4_swiglu_q4", "grouped_gemm_fp8", "moe_router_topk", "moe_dispatch", "moe_finalize", "moe_combine", "moe_rows_bound", "device_status",
    "clear_device_status", "BSError", "EPI_STORE", "EPI_SWIGLU", "EPI_COMBINE", "EPI_ROWS", "kernel_options",
    "current_kernel_options", "FP4_ONE_CTA", "FP4_PAIR",
]

BS_OK, BS_ERR_INVALID, BS_ERR_ALIGN, BS_ERR_UNSUPPORTED, BS_ERR_CUDA, BS_ERR_TIMEOUT, BS_ERR_OFFSETS = range(7)
DTYPE_F32, DTYPE_BF16 = 0, 1
FMT_FP4, FMT_FP8 = 0, 1
EPI_STORE, EPI_SWIGLU, EPI_COMBINE, EPI_ROWS = 0, 1, 2, 3
Q8_TOKEN, Q8_BLOCK, Q8_ROW = 1, 128, 3


class BSError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"bsgemm status {status}: {msg}")
        self.status = status


class GemmArgs(ctypes.Structure):
    _fields_ = [
        ("fmt", ctypes.c_int), ("a", ctypes.c_void_p), ("sfa", ctypes.c_void_p), ("b", ctypes.c_void_p),
        ("sfb", ctypes.c_void_p), ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
        ("alpha", ctypes.c_float), ("col_scale", ctypes.c_void_p), ("lora_t", ctypes.c_void_p),
        ("lora_b_t", ctypes.c_void_p), ("r", ctypes.c_int), ("bias", ctypes.c_void_p), ("out", ctypes.c_void_p),
        ("out_dtype", ctypes.c_int), ("ldo", ctypes.c_int64), ("num_sms", ctypes.c_int),
        ("n_chunk_blocks", ctypes.c_int), ("fp4_kernel", ctypes.c_int), ("fp4_stage_k", ctypes.c_int),
        ("fp4_small_experts", ctypes.c_int), ("fp4_half_tail", ctypes.c_int), ("fp8_stream_k", ctypes.c_int),
        ("fp8_scaling", ctypes.c_int), ("wait_timeout_us", ctypes.c_int), ("weights_ready", ctypes.c_int), ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t), ("a_tensor_scale", ctypes.c_void_p), ("b_tensor_scale", ctypes.c_void_p),
        ("fp4_decode", ctypes.c_int),
    ]


# Per-call kernel choices of bs_gemm_args (0 = the library's default), see
# include/bsgemm.h.  Every GEMM call of this binding fills them from the
# options active on the calling thread: the defaults, or those of an enclosing
# ``with kernel_options(...)`` block.
_CHOICES = ("fp4_kernel", "fp4_stage_k", "fp4_small_experts", "fp4_half_tail", "fp4_decode", "fp8_stream_k",
            "wait_timeout_us")
FP4_ONE_CTA, FP4_PAIR = 1, 2
_tls = threading.local()


def current_kernel_options() -> dict:
    return dict(getattr(_tls, "opts", {}))


class kernel_options:
    """Context manager: GEMM calls made on this thread inside the block pass
    these kernel choices in their bs_gemm_args (unnamed fields keep the value
    of any enclosing block, else 0 = default)."""

    def __init__(self, **choices):
        bad = set(choices) - set(_CHOICES)
        if bad:
            raise TypeError(f"unknown kernel choices {sorted(bad)}")
        self.choices = {k: int(v) for k, v in choices.items()}

    def __enter__(self):
        self.saved = getattr(_tls, "opts", {})
        _tls.opts = {**self.saved, **self.choices}
        return self

    def __exit__(self, *exc):
        _tls.opts = self.saved
        return False


_lib = None
_lock = threading.Lock()


def load(path: str | None = None):
    """Load libbsgemm.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or os.environ.get("BSGEMM_LIB") or _LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"CUDA library not built: {p} is missing (run __graft_entry__.build())")
        lib = ctypes.CDLL(p)
        P, I64, I, F, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.bs_sf_bytes.restype = SZ
        lib.bs_sf_bytes.argtypes = [I64, I64]
        lib.bs_sf_offset.restype = I64
        lib.bs_sf_offset.argtypes = [I64, I64, I64]
        lib.q4_quantize.restype = I
        lib.q4_quantize.argtypes = [P, I, I64, I64, I64, P, P, P, P, I, P, P]
        lib.bs_tensor_amax.restype = I
        lib.bs_tensor_amax.argtypes = [P, I, I64, I64, I64, P, P]
        lib.q4_quantize_two_level.restype = I
        lib.q4_quantize_two_level.argtypes = [P, I, I64, I64, I64, P, P, P, P, P]
        lib.bs_fp4_gather_rows.restype = I
        lib.bs_fp4_gather_rows.argtypes = [P, P, I64, I64, P, I64, P, P, P]
        lib.bs_fp8_gather_rows.restype = I
        lib.bs_fp8_gather_rows.argtypes = [P, P, I64, I64, P, I64, P, P, P]
        lib.q8_quantize.restype = I
        lib.q8_quantize.argtypes = [P, I, I64, I64, I64, I, P, P, P]
        lib.bs_gemm.restype = I
        lib.bs_gemm.argtypes = [ctypes.POINTER(GemmArgs), P]
        lib.bs_gemm_workspace_bytes.restype = SZ
        lib.bs_gemm_workspace_bytes.argtypes = [ctypes.POINTER(GemmArgs)]
        lib.bs_gemm_multi.restype = I
        lib.bs_gemm_multi.argtypes = [ctypes.POINTER(GemmArgs), I, P, P, P, P]
        lib.bs_gemm_multi_workspace_bytes.restype = SZ
        lib.bs_gemm_multi_workspace_bytes.argtypes = [ctypes.POINTER(GemmArgs), I]
        lib.bs_grouped_gemm.restype = I
        lib.bs_grouped_gemm.argtypes = [ctypes.POINTER(GemmArgs), I, P, P, I, P, P, P, I64, P]
        lib.bs_moe_rows_bound.restype = I64
        lib.bs_grouped_gemm_swiglu_q4.restype = I
        lib.bs_grouped_gemm_swiglu_q4.argtypes = [ctypes.POINTER(GemmArgs), I, P, P, P, P, P]
        lib.bs_moe_rows_bound.argtypes = [I64, I, I]
        lib.bs_moe_dispatch_workspace_bytes.restype = SZ
        lib.bs_moe_dispatch_workspace_bytes.argtypes = [I64, I, I]
        lib.bs_moe_router_topk.restype = I
        lib.bs_moe_router_topk.argtypes = [P, I64, I, I, P, P, P]
        lib.bs_moe_dispatch.restype = I
        lib.bs_moe_dispatch.argtypes = [P, P, I64, I, I, P, P, P, P, P, P, SZ, P]
        lib.bs_moe_dispatch_noalloc.restype = I
        lib.bs_moe_dispatch_noalloc.argtypes = [P, P, I64, I, I, P, P, P, P, P, P]
        lib.bs_moe_finalize.restype = I
        lib.bs_moe_finalize.argtypes = [P, P, I64, P]
        lib.bs_moe_combine.restype = I
        lib.bs_moe_combine.argtypes = [P, I64, P, I64, I64, I, I64, P, P, I64, P]
        lib.bs_get_device_status.restype = I
        lib.bs_get_device_status.argtypes = [ctypes.POINTER(I)]
        lib.bs_clear_device_status.restype = I
        lib.bs_clear_device_status.argtypes = []
        lib.bs_status_string.restype = ctypes.c_char_p
        lib.bs_status_string.argtypes = [I]
        lib.bs_last_error.restype = ctypes.c_char_p
        lib.bs_last_error.argtypes = []
        _ = F
        _lib = lib
        return lib


def _check(status: int):
    if status != BS_OK:
        lib = load()
        raise BSError(status, lib.bs_last_error().decode(errors="replace") or
                      lib.bs_status_string(status).decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return DTYPE_F32
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def sf_bytes(rows: int, K: int) -> int:
    """Bytes of the MMA-layout scale tensor of an [rows, K] FP4 operand."""
    return int(load().bs_sf_bytes(rows, K))


def sf_offset(row: int, group: int, K: int) -> int:
    return int(load().bs_sf_offset(row, group, K))


def q4_quantize(x: torch.Tensor, gather: torch.Tensor | None = None, rows: int | None = None,
                lora_a_t: torch.Tensor | None = None, out=None, stream=None):
    """FP4 E2M1 group-16 quantization.  Returns (codes [M, K/2] u8, sf u8 [sf_bytes],
    lora_t bf16 [M, 64] or None).  With ``gather``, output row i is x[gather[i]]
    (negative: zero row) and M = len(gather) (or ``rows``)."""
    assert x.is_cuda and x.dim() == 2 and x.stride(1) == 1
    M = int(rows if rows is not None else (gather.numel() if gather is not None else x.shape[0]))
    K = x.shape[1]
    if out is None:
        codes = torch.empty((M, K // 2), dtype=torch.uint8, device=x.device)
        sf = torch.empty(sf_bytes(M, K), dtype=torch.uint8, device=x.device)
        lt = torch.empty((M, 64), dtype=torch.bfloat16, device=x.device) if lora_a_t is not None else None
    else:
        codes, sf, lt = out
    _check(load().q4_quantize(_ptr(x), _dt(x), M, K, x.stride(0), _ptr(gather), _ptr(codes), _ptr(sf),
                              _ptr(lora_a_t), 32 if lora_a_t is not None else 0, _ptr(lt), _stream(stream)))
    return codes, sf, lt


def tensor_amax(x: torch.Tensor, out=None, stream=None):
    """max |x| over the whole [M, K] tensor, as a device fp32 tensor [1]."""
    amax = out if out is not None else torch.empty(1, dtype=torch.float32, device=x.device)
    _check(load().bs_tensor_amax(_ptr(x), _dt(x), x.shape[0], x.shape[1], x.stride(0), _ptr(amax), _stream(stream)))
    return amax


def q4_quantize_two_level(x: torch.Tensor, amax=None, out=None, stream=None):
    """Two-level FP4: power-of-two tensor scale above the e4m3 group scales.
    Returns (codes [M, K/2], sf, tensor_scale device fp32 [1]); ``amax``
    (device fp32 [1]) defaults to tensor_amax(x)."""
    assert x.is_cuda and x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    if amax is None:
        amax = tensor_amax(x, stream=stream)
    if out is None:
        out = (torch.empty((M, K // 2), dtype=torch.uint8, device=x.device),
               torch.empty(sf_bytes(M, K), dtype=torch.uint8, device=x.device),
               torch.empty(1, dtype=torch.float32, device=x.device))
    codes, sf, ts = out
    _check(load().q4_quantize_two_level(_ptr(x), _dt(x), M, K, x.stride(0), _ptr(amax), _ptr(codes), _ptr(sf),
                                        _ptr(ts), _stream(stream)))
    return codes, sf, ts


def fp4_gather_rows(codes, sf, K: int, gather, out=None, stream=None):
    """Rows gather[i] of an FP4 matrix (codes + MMA-layout scales); -1 -> zero row."""
    rows_out = gather.numel()
    if out is None:
        out = (torch.empty((rows_out, K // 2), dtype=torch.uint8, device=codes.device),
               torch.empty(sf_bytes(rows_out, K), dtype=torch.uint8, device=codes.device))
    _check(load().bs_fp4_gather_rows(_ptr(codes), _ptr(sf), codes.shape[0], K, _ptr(gather), rows_out,
                                     _ptr(out[0]), _ptr(out[1]), _stream(stream)))
    return out


def fp8_gather_rows(codes, scales, gather, out=None, stream=None):
    """Rows gather[i] of an FP8 matrix (codes [rows, K] + TOKEN-mode scales
    [K/128, rows]); -1 -> zero row with zero scales."""
    rows_in, K = codes.shape
    rows_out = gather.numel()
    if out is None:
        out = (torch.empty((rows_out, K), dtype=torch.uint8, device=codes.device),
               torch.empty((K // 128, rows_out), dtype=torch.float32, device=codes.device))
    _check(load().bs_fp8_gather_rows(_ptr(codes), _ptr(scales), rows_in, K, _ptr(gather), rows_out,
                                     _ptr(out[0]), _ptr(out[1]), _stream(stream)))
    return out


def q8_quantize(x: torch.Tensor, mode: int = Q8_TOKEN, out=None, stream=None):
    """FP8 e4m3 quantization.  TOKEN mode: scales fp32 [K/128, M]; BLOCK mode:
    scales fp32 [ceil(M/128), K/128]; ROW mode (W8A8): scales fp32 [M]."""
    assert x.is_cuda and x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    if out is None:
        codes = torch.empty((M, K), dtype=torch.uint8, device=x.device)
        shape = {Q8_TOKEN: (K // 128, M), Q8_BLOCK: ((M + 127) // 128, K // 128), Q8_ROW: (M,)}[mode]
        scales = torch.empty(shape, dtype=torch.float32, device=x.device)
    else:
        codes, scales = out
    _check(load().q8_quantize(_ptr(x), _dt(x), M, K, x.stride(0), mode, _ptr(codes), _ptr(scales),
                              _stream(stream)))
    return codes, scales


def _args(fmt, a, sfa, b, sfb, M, N, K, out, alpha=1.0, col_scale=None, lora_t=None, lora_b_t=None,
          bias=None, num_sms=0):
    g = GemmArgs()
    g.fmt = fmt
    g.a, g.sfa, g.b, g.sfb = a.data_ptr(), sfa.data_ptr(), b.data_ptr(), sfb.data_ptr()
    g.M, g.N, g.K = M, N, K
    g.alpha = alpha
    g.col_scale = None if col_scale is None else col_scale.data_ptr()
    g.lora_t = None if lora_t is None else lora_t.data_ptr()
    g.lora_b_t = None if lora_b_t is None else lora_b_t.data_ptr()
    g.r = 32 if lora_t is not None else 0
    g.bias = None if bias is None else bias.data_ptr()
    if out is not None:
        g.out = out.data_ptr()
        g.out_dtype = _dt(out)
        g.ldo = out.stride(0)
    g.num_sms = num_sms
    for k, v in getattr(_tls, "opts", {}).items():
        setattr(g, k, v)
    return g


def gemm_fp4(a, sfa, b, sfb, K: int, out_dtype=torch.bfloat16, alpha: float = 1.0, col_scale=None,
             lora_t=None, lora_b_t=None, bias=None, out=None, num_sms: int = 0, a_tensor_scale=None,
             b_tensor_scale=None, weights_ready: bool = False, stream=None):
    """Dense block-scaled FP4 GEMM: Y[M, N] from A codes [M, K/2] and B codes [N, K/2]
    (two-level operands: their device tensor scales from q4_quantize_two_level)."""
    M, N = a.shape[0], b.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=a.device)
    g = _args(FMT_FP4, a, sfa, b, sfb, M, N, K, out, alpha, col_scale, lora_t, lora_b_t, bias, num_sms)
    g.a_tensor_scale = None if a_tensor_scale is None else a_tensor_scale.data_ptr()
    g.b_tensor_scale = None if b_tensor_scale is None else b_tensor_scale.data_ptr()
    g.weights_ready = 1 if weights_ready else 0
    lib = load()
    nbytes = int(lib.bs_gemm_workspace_bytes(ctypes.byref(g)))
    if nbytes:   # the decode kernel (M <= 32): stream-K scratch
        s = stream if stream is not None else torch.cuda.current_stream(a.device)
        ws = _workspace(a.device, s, nbytes)
        g.workspace, g.workspace_bytes = ws.data_ptr(), ws.numel()
    _check(load().bs_gemm(ctypes.byref(g), _stream(stream)))
    return out


# Workspaces of the FP8 stream-K schedule, one per (device, stream): calls on
# one stream run in order, so they may share it; the library leaves it zeroed
# where the next call reads it.
_workspaces: dict = {}


def _workspace(device, stream, nbytes: int):
    key = (device.index, stream.cuda_stream)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def gemm_fp8(a, sa, b, sb, out_dtype=torch.bfloat16, out=None, num_sms: int = 0, weights_ready: bool = False,
             rowwise: bool = False, stream=None):
    """Dense FP8 GEMM with 1x128 A scales [K/128, M] and 128x128 B scales.
    ``weights_ready``: the kernel just before this call on the stream does not
    write ``b`` / ``sb``, so the weight loads may start before it finishes."""
    M, K = a.shape
    N = b.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=a.device)
    g = _args(FMT_FP8, a, sa, b, sb, M, N, K, out, num_sms=num_sms)
    g.weights_ready = 1 if weights_ready else 0
    g.fp8_scaling = 2 if rowwise else 0   # W8A8: sa [M] per token, sb [N] per channel
    lib = load()
    nbytes = int(lib.bs_gemm_workspace_bytes(ctypes.byref(g)))
    if nbytes:
        s = stream if stream is not None else torch.cuda.current_stream(a.device)
        ws = _workspace(a.device, s, nbytes)
        g.workspace, g.workspace_bytes = ws.data_ptr(), ws.numel()
    _check(lib.bs_gemm(ctypes.byref(g), _stream(stream)))
    return out


def _gemm_multi(fmt, a, sa, weights, M, N, K, out_dtype, outs, num_sms, weights_ready, alpha=1.0,
                a_tensor_scale=None, stream=None):
    G = len(weights)
    if G == 0:
        raise ValueError("bs_gemm_multi needs at least one weight set")
    if outs is not None and len(outs) != G:
        raise ValueError(f"{len(outs)} outputs for {G} weight sets")
    if outs is None:
        outs = [torch.empty((M, N), dtype=out_dtype, device=a.device) for _ in range(G)]
    b0, sb0 = weights[0]
    g = _args(fmt, a, sa, b0, sb0, M, N, K, outs[0], alpha=alpha, num_sms=num_sms)
    g.weights_ready = 1 if weights_ready else 0
    g.a_tensor_scale = None if a_tensor_scale is None else a_tensor_scale.data_ptr()
    arr = ctypes.c_void_p * max(G, 1)
    bp = arr(*[w[0].data_ptr() for w in weights])
    sp = arr(*[w[1].data_ptr() for w in weights])
    op = arr(*[o.data_ptr() for o in outs])
    lib = load()
    nbytes = int(lib.bs_gemm_multi_workspace_bytes(ctypes.byref(g), G))
    if nbytes:
        s = stream if stream is not None else torch.cuda.current_stream(a.device)
        ws = _workspace(a.device, s, nbytes)
        g.workspace, g.workspace_bytes = ws.data_ptr(), ws.numel()
    _check(lib.bs_gemm_multi(ctypes.byref(g), G, bp, sp, op, _stream(stream)))
    return outs


def gemm_fp8_multi(a, sa, weights, out_dtype=torch.bfloat16, outs=None, num_sms: int = 0,
                   weights_ready: bool = False, stream=None):
    """G block-scaled FP8 GEMMs that share the tokens ``a`` [M, K] (M <= 32,
    TOKEN-mode scales ``sa``) in one launch: ``weights`` is a list of (codes
    [N, K], BLOCK-mode scales) pairs, one per product; returns the G outputs
    [M, N] (or fills ``outs``)."""
    M, K = a.shape
    N = weights[0][0].shape[0] if weights else 0
    return _gemm_multi(FMT_FP8, a, sa, weights, M, N, K, out_dtype, outs, num_sms, weights_ready, stream=stream)


def gemm_fp4_multi(a, sfa, weights, K: int, out_dtype=torch.bfloat16, outs=None, alpha: float = 1.0,
                   a_tensor_scale=None, num_sms: int = 0, weights_ready: bool = False, stream=None):
    """G FP4 decode GEMMs that share the tokens ``a`` (codes [M, K/2], M <= 32,
    scales ``sfa``) in one launch: ``weights`` is a list of (codes [N, K/2],
    scales) pairs from q4_quantize; returns the G outputs [M, N]."""
    M = a.shape[0]
    N = weights[0][0].shape[0] if weights else 0
    return _gemm_multi(FMT_FP4, a, sfa, weights, M, N, K, out_dtype, outs, num_sms, weights_ready, alpha=alpha,
                       a_tensor_scale=a_tensor_scale, stream=stream)


def grouped_gemm_fp4(a, sfa, b, sfb, K: int, N: int, E: int, offsets, counts, epilogue: int, out=None,
                     token_of=None, weight_of=None, out32=None, num_sms: int = 0, n_chunk_blocks: int = 0,
                     stream=None):
    """FP4 GEMM grouped over experts (rows of ``a`` grouped by ``offsets``/``counts``)."""
    M = a.shape[0]
    g = _args(FMT_FP4, a, sfa, b, sfb, M, N, K, out, num_sms=num_sms)
    g.n_chunk_blocks = n_chunk_blocks
    ld32 = 0 if out32 is None else out32.stride(0)
    _check(load().bs_grouped_gemm(ctypes.byref(g), E, _ptr(offsets), _ptr(counts), epilogue, _ptr(token_of),
                                  _ptr(weight_of), _ptr(out32), ld32, _stream(stream)))
    return out


def grouped_gemm_fp8(a, sfa, b, sfb, N: int, E: int, offsets, counts, epilogue: int, out=None, weight_of=None,
                     num_sms: int = 0, stream=None):
    """FP8 GEMM grouped over experts: ``a`` e4m3 [M, K] with TOKEN-mode scales
    ``sfa`` [K/128, M] (rows grouped by ``offsets``/``counts``), ``b`` the
    stacked expert weights [E*Nw, K] with 128x128 block scales ``sfb``.
    Epilogues EPI_STORE, EPI_SWIGLU (bf16 h) and EPI_ROWS (fp32, weight_of)."""
    M, K = a.shape
    if out is None:
        dt = torch.float32 if epilogue == EPI_ROWS else torch.bfloat16
        out = torch.empty((M, N), dtype=dt, device=a.device)
    g = _args(FMT_FP8, a, sfa, b, sfb, M, N, K, out, num_sms=num_sms)
    _check(load().bs_grouped_gemm(ctypes.byref(g), E, _ptr(offsets), _ptr(counts), epilogue, None,
                                  _ptr(weight_of), None, 0, _stream(stream)))
    return out


def grouped_gemm_fp4_swiglu_q4(a, sfa, b, sfb, K: int, N: int, E: int, offsets, counts, h_codes=None, h_sf=None,
                               num_sms: int = 0, n_chunk_blocks: int = 0, stream=None):
    """Grouped gate/up GEMM with h = bf16(silu(g) * u) quantized to FP4 in the
    epilogue: returns (h_codes uint8 [M, N/2], h_sf scale bytes), as
    q4_quantize would write them for the segment rows."""
    M = a.shape[0]
    if h_codes is None:
        h_codes = torch.empty((M, N // 2), dtype=torch.uint8, device=a.device)
    if h_sf is None:
        h_sf = torch.empty(sf_bytes(M, N), dtype=torch.uint8, device=a.device)
    g = _args(FMT_FP4, a, sfa, b, sfb, M, N, K, None, num_sms=num_sms)
    g.n_chunk_blocks = n_chunk_blocks
    _check(load().bs_grouped_gemm_swiglu_q4(ctypes.byref(g), E, _ptr(offsets), _ptr(counts), _ptr(h_codes),
                                            _ptr(h_sf), _stream(stream)))
    return h_codes, h_sf


def moe_rows_bound(T: int, k: int, E: int) -> int:
    return int(load().bs_moe_rows_bound(T, k, E))


def moe_router_topk(logits, k: int, out=None, stream=None):
    """Top-k routing from fp32 router logits [T, E]: (topk_ids int32 [T, k] in
    descending order of logit, ties to the lower id; topk_w fp32 [T, k], the
    softmax of the chosen logits)."""
    T, E = logits.shape
    if out is None:
        out = (torch.empty((T, k), dtype=torch.int32, device=logits.device),
               torch.empty((T, k), dtype=torch.float32, device=logits.device))
    _check(load().bs_moe_router_topk(_ptr(logits), T, E, k, _ptr(out[0]), _ptr(out[1]), _stream(stream)))
    return out


def moe_dispatch(topk_ids, topk_w, E: int, out=None, workspace=None, stream=None):
    """Group (token, slot) pairs by expert.  Returns dict(counts, offsets,
    pair_of_row, token_of, weight_of) of device tensors (rows = moe_rows_bound)."""
    lib = load()
    T, k = topk_ids.shape
    dev = topk_ids.device
    rows = moe_rows_bound(T, k, E)
    if out is None:
        out = dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
                   offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                   pair_of_row=torch.empty(rows, dtype=torch.int32, device=dev),
                   token_of=torch.empty(rows, dtype=torch.int32, device=dev),
                   weight_of=torch.empty(rows, dtype=torch.float32, device=dev))
    wsb = int(lib.bs_moe_dispatch_workspace_bytes(T, k, E))
    if workspace is None:
        workspace = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
    _check(lib.bs_moe_dispatch(_ptr(topk_ids), _ptr(topk_w), T, k, E, _ptr(out["counts"]), _ptr(out["offsets"]),
                               _ptr(out["pair_of_row"]), _ptr(out["token_of"]), _ptr(out["weight_of"]),
                               _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def moe_finalize(out32, out_bf16, stream=None):
    _check(load().bs_moe_finalize(_ptr(out32), _ptr(out_bf16), out32.numel(), _stream(stream)))
    return out_bf16


def moe_combine(rows, pair_of_row, T: int, k: int, out=None, row_of_pair=None, stream=None):
    """out[t] = bf16(sum_j rows[row of pair t*k + j]) (fp32 sum in slot order);
    ``rows`` fp32 [n_rows, H] from a grouped GEMM with EPI_ROWS."""
    n_rows, H = rows.shape
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=rows.device)
    if row_of_pair is None:
        row_of_pair = torch.empty(max(T * k, 1), dtype=torch.int32, device=rows.device)
    _check(load().bs_moe_combine(_ptr(rows), rows.stride(0), _ptr(pair_of_row), n_rows, T, k, H, _ptr(row_of_pair),
                                 _ptr(out), out.stride(0), _stream(stream)))
    return out


def device_status() -> tuple[int, int]:
    d = ctypes.c_int(0)
    s = load().bs_get_device_status(ctypes.byref(d))
    return int(s), int(d.value)


def clear_device_status():
    _check(load().bs_clear_device_status())
