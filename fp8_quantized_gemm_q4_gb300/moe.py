"""Grouped FP4 and FP8 MoE layers composed from the library's entry points.

Order of the layer ("DeepGEMM for Hopper MoE", sections 1 and 3; "DeepGEMM
teardown (FP8 GEMM)", section 5.3):

  0. bs_moe_router_topk  (forward_logits) top-k experts of every token from
                         its router logits, softmax weights of the chosen
  1. bs_moe_dispatch     group the (token, slot) pairs by expert into
                         128-aligned contiguous segments
  2. q4_quantize         quantize each token's row once (online), then
     bs_fp4_gather_rows  gather the quantized rows into the expert segments
                         (bit-identical to quantizing the gathered rows)
  3. bs_grouped_gemm_swiglu_q4
                         gate/up GEMM per expert whose epilogue forms
                         h = bf16(silu(x W_gate^T) * (x W_up^T)) and
  4.                     re-quantizes it to FP4 in place ("DeepGEMM for
                         Hopper MoE", section 3: h never goes through memory
                         as bf16); h_quant="separate" runs the SWIGLU
                         epilogue (bf16 h) and q4_quantize instead
  5. bs_grouped_gemm     down GEMM per expert; the routed combine ("Blackwell
                         FP4 MoE TFLOPS optimisation", section 3.2, result
                         aggregation) runs one of two ways:
       combine="rows"    (default) the GEMM writes each row's weighted result
                         w * (h W_down^T) in fp32 (coalesced TMA stores), then
     6. bs_moe_combine   sums each token's k rows in slot order -> bf16 out
                         (deterministic; no atomics)
       combine="atomic"  the GEMM reduces w * (h W_down^T) into out32[token]
     6. bs_moe_finalize  (fp32 reductions at L2), then out = bf16(out32) and
                         out32 is reset to zero

The FP8 layer (Fp8MoELayer; "DeepGEMM teardown (FP8 GEMM)", sections 2.2 and
5.3; "DeepGEMM for Hopper MoE", section 2.1) runs the same order in e4m3 with
fp32 scales per 1x128 token block (x and h) and per 128x128 block of the
stacked expert weights: router, dispatch, q8_quantize + bs_fp8_gather_rows,
the grouped FP8 gate/up GEMM with the SWIGLU epilogue (bf16 h), q8_quantize
of h, the grouped FP8 down GEMM with the ROWS epilogue, bs_moe_combine.

Every step is one or more of the library's kernels; this module only holds
the buffers and calls them in order.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import (EPI_COMBINE, EPI_ROWS, EPI_SWIGLU, Q8_BLOCK, Q8_TOKEN, fp4_gather_rows, fp8_gather_rows,
               grouped_gemm_fp4, grouped_gemm_fp4_swiglu_q4, grouped_gemm_fp8, moe_combine, moe_dispatch,
               moe_finalize, moe_router_topk, moe_rows_bound, q4_quantize, q8_quantize, sf_bytes)


@dataclass
class MoEWeights:
    """Stacked FP4 expert weights: gate/up [E*2F, H] (gate rows first per
    expert) and down [E*H, F], codes plus MMA-layout scales."""
    E: int
    H: int
    F: int
    wgu_codes: torch.Tensor
    wgu_sf: torch.Tensor
    wd_codes: torch.Tensor
    wd_sf: torch.Tensor


def quantize_expert_weights(wgu_list, wd_list, device="cuda") -> MoEWeights:
    """Quantize per-expert bf16 weights (offline, outside the layer's timed path)."""
    E = len(wgu_list)
    F2, H = wgu_list[0].shape
    F = F2 // 2
    wgu_codes = torch.empty((E * F2, H // 2), dtype=torch.uint8, device=device)
    wgu_sf = torch.empty(sf_bytes(E * F2, H), dtype=torch.uint8, device=device)
    wd_codes = torch.empty((E * H, F // 2), dtype=torch.uint8, device=device)
    wd_sf = torch.empty(sf_bytes(E * H, F), dtype=torch.uint8, device=device)
    per_gu, per_d = sf_bytes(F2, H), sf_bytes(H, F)
    for e in range(E):
        wgu = wgu_list[e].to(device)
        wd = wd_list[e].to(device)
        q4_quantize(wgu, out=(wgu_codes[e * F2:(e + 1) * F2], wgu_sf[e * per_gu:(e + 1) * per_gu], None))
        q4_quantize(wd, out=(wd_codes[e * H:(e + 1) * H], wd_sf[e * per_d:(e + 1) * per_d], None))
    return MoEWeights(E, H, F, wgu_codes, wgu_sf, wd_codes, wd_sf)


@dataclass
class Fp8MoEWeights:
    """Stacked FP8 expert weights: e4m3 gate/up [E*2F, H] (gate rows first per
    expert) and down [E*H, F], with the fp32 128x128 block scales of the
    stacked matrices ([E*2F/128, H/128] and [E*H/128, F/128])."""
    E: int
    H: int
    F: int
    wgu_codes: torch.Tensor
    wgu_sf: torch.Tensor
    wd_codes: torch.Tensor
    wd_sf: torch.Tensor


def quantize_expert_weights_fp8(wgu_list, wd_list, device="cuda") -> Fp8MoEWeights:
    """Quantize per-expert bf16 weights to FP8 with 128x128 block scales
    (offline, outside the layer's timed path).  2F and H are multiples of
    128, so the blocks of one expert are exactly its rows of the stacked scales."""
    E = len(wgu_list)
    F2, H = wgu_list[0].shape
    F = F2 // 2
    wgu_codes = torch.empty((E * F2, H), dtype=torch.uint8, device=device)
    wgu_sf = torch.empty((E * F2 // 128, H // 128), dtype=torch.float32, device=device)
    wd_codes = torch.empty((E * H, F), dtype=torch.uint8, device=device)
    wd_sf = torch.empty((E * H // 128, F // 128), dtype=torch.float32, device=device)
    bg, bd = F2 // 128, H // 128
    for e in range(E):
        q8_quantize(wgu_list[e].to(device), mode=Q8_BLOCK,
                    out=(wgu_codes[e * F2:(e + 1) * F2], wgu_sf[e * bg:(e + 1) * bg]))
        q8_quantize(wd_list[e].to(device), mode=Q8_BLOCK,
                    out=(wd_codes[e * H:(e + 1) * H], wd_sf[e * bd:(e + 1) * bd]))
    return Fp8MoEWeights(E, H, F, wgu_codes, wgu_sf, wd_codes, wd_sf)


class _GraphedLayer:
    """Router entry, CUDA-graph capture and replay shared by the FP4 and FP8
    layers.  A subclass sets T, k, the topk_ids / topk_w / out buffers and
    implements forward(x, topk_ids, topk_w)."""

    def _routing_buffers(self, T: int, k: int, device):
        self.topk_ids = torch.empty((T, k), dtype=torch.int32, device=device)
        self.topk_w = torch.empty((T, k), dtype=torch.float32, device=device)

    def forward(self, x: torch.Tensor, topk_ids: torch.Tensor, topk_w: torch.Tensor) -> torch.Tensor:
        raise NotImplementedError

    def forward_logits(self, x: torch.Tensor, logits: torch.Tensor) -> torch.Tensor:
        """The layer from the router's fp32 logits [T, E]: top-k routing on the
        GPU, then forward()."""
        moe_router_topk(logits, self.k, out=(self.topk_ids, self.topk_w))
        return self.forward(x, self.topk_ids, self.topk_w)

    def capture(self, x: torch.Tensor, topk_ids: torch.Tensor | None = None, topk_w: torch.Tensor | None = None,
                logits: torch.Tensor | None = None) -> None:
        """Record the whole layer (all its launches) as one CUDA graph ("Blackwell
        FP4 MoE TFLOPS optimisation", section 3.2: the compute flow captured in a
        CUDA Graph), from the routing or, given ``logits``, from the router.
        The graph reads static copies of the inputs; replay() refreshes them and
        runs the layer with one graph launch."""
        self.static_x = x.clone()
        self.static_logits = None if logits is None else logits.clone()
        self.static_ids = None if topk_ids is None else topk_ids.clone()
        self.static_w = None if topk_w is None else topk_w.clone()

        def run():
            if self.static_logits is not None:
                self.forward_logits(self.static_x, self.static_logits)
            else:
                self.forward(self.static_x, self.static_ids, self.static_w)

        run()  # sizes the dispatch tables
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                run()
        torch.cuda.current_stream().wait_stream(side)
        self.graph = g

    def replay(self, x: torch.Tensor | None = None, topk_ids: torch.Tensor | None = None,
               topk_w: torch.Tensor | None = None, logits: torch.Tensor | None = None) -> torch.Tensor:
        """Run the captured layer; given inputs are first copied into the static ones."""
        for src, dst in ((x, self.static_x), (topk_ids, self.static_ids), (topk_w, self.static_w),
                         (logits, self.static_logits)):
            if src is not None:
                dst.copy_(src, non_blocking=True)
        self.graph.replay()
        return self.out


class MoELayer(_GraphedLayer):
    """FP4 layer.  Holds the per-call buffers of one layer shape so repeated
    calls (and a CUDA-graph capture) allocate nothing."""

    def __init__(self, weights: MoEWeights, T: int, k: int, device="cuda", combine: str = "rows",
                 h_quant: str = "fused"):
        if combine not in ("rows", "atomic"):
            raise ValueError(f"combine must be 'rows' or 'atomic', not {combine!r}")
        if h_quant not in ("fused", "separate"):
            raise ValueError(f"h_quant must be 'fused' or 'separate', not {h_quant!r}")
        self.w = weights
        self.T, self.k = T, k
        self.combine = combine
        self.h_quant = h_quant
        E, H, F = weights.E, weights.H, weights.F
        self.rows = moe_rows_bound(T, k, E)
        self.tq = torch.empty((T, H // 2), dtype=torch.uint8, device=device)
        self.ts = torch.empty(sf_bytes(T, H), dtype=torch.uint8, device=device)
        self.xq = torch.empty((self.rows, H // 2), dtype=torch.uint8, device=device)
        self.xs = torch.empty(sf_bytes(self.rows, H), dtype=torch.uint8, device=device)
        # bf16 h only on the separate path
        self.h = torch.zeros((self.rows, F), dtype=torch.bfloat16, device=device) if h_quant == "separate" else None
        self.hq = torch.empty((self.rows, F // 2), dtype=torch.uint8, device=device)
        self.hs = torch.empty(sf_bytes(self.rows, F), dtype=torch.uint8, device=device)
        if combine == "rows":
            self.yrows = torch.empty((self.rows, H), dtype=torch.float32, device=device)
            self.row_of_pair = torch.empty(max(T * k, 1), dtype=torch.int32, device=device)
        else:
            self.out32 = torch.zeros((T, H), dtype=torch.float32, device=device)
        # Atomic combine tile order: chunks of 256-column blocks small enough
        # that the fp32 accumulator slab they reduce into (T x 256 x 4 bytes
        # per block) stays within about half of the 129 MB L2.
        self.combine_chunk = max(1, (64 << 20) // (T * 256 * 4))
        self.out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        # routing of forward_logits (the router's outputs, the dispatch's inputs)
        self._routing_buffers(T, k, device)
        self.disp = None
        from . import load
        wsb = int(load().bs_moe_dispatch_workspace_bytes(T, k, E))
        self.workspace = torch.empty(max(wsb, 16), dtype=torch.uint8, device=device)

    def forward(self, x: torch.Tensor, topk_ids: torch.Tensor, topk_w: torch.Tensor) -> torch.Tensor:
        w = self.w
        self.disp = moe_dispatch(topk_ids, topk_w, w.E, out=self.disp, workspace=self.workspace)
        d = self.disp
        q4_quantize(x, out=(self.tq, self.ts, None))
        fp4_gather_rows(self.tq, self.ts, w.H, d["token_of"], out=(self.xq, self.xs))
        if self.h_quant == "fused":
            grouped_gemm_fp4_swiglu_q4(self.xq, self.xs, w.wgu_codes, w.wgu_sf, K=w.H, N=w.F, E=w.E,
                                       offsets=d["offsets"], counts=d["counts"], h_codes=self.hq, h_sf=self.hs)
        else:
            grouped_gemm_fp4(self.xq, self.xs, w.wgu_codes, w.wgu_sf, K=w.H, N=w.F, E=w.E, offsets=d["offsets"],
                             counts=d["counts"], epilogue=EPI_SWIGLU, out=self.h)
            q4_quantize(self.h, out=(self.hq, self.hs, None))
        if self.combine == "rows":
            grouped_gemm_fp4(self.hq, self.hs, w.wd_codes, w.wd_sf, K=w.F, N=w.H, E=w.E, offsets=d["offsets"],
                             counts=d["counts"], epilogue=EPI_ROWS, out=self.yrows, weight_of=d["weight_of"])
            moe_combine(self.yrows, d["pair_of_row"], self.T, self.k, out=self.out, row_of_pair=self.row_of_pair)
        else:
            grouped_gemm_fp4(self.hq, self.hs, w.wd_codes, w.wd_sf, K=w.F, N=w.H, E=w.E, offsets=d["offsets"],
                             counts=d["counts"], epilogue=EPI_COMBINE, token_of=d["token_of"],
                             weight_of=d["weight_of"], out32=self.out32, n_chunk_blocks=self.combine_chunk)
            moe_finalize(self.out32, self.out)
        return self.out


class Fp8MoELayer(_GraphedLayer):
    """FP8 layer (e4m3, 1x128 token and 128x128 weight-block fp32 scales).
    Holds the per-call buffers of one layer shape so repeated calls (and a
    CUDA-graph capture) allocate nothing."""

    def __init__(self, weights: Fp8MoEWeights, T: int, k: int, device="cuda"):
        self.w = weights
        self.T, self.k = T, k
        E, H, F = weights.E, weights.H, weights.F
        self.rows = moe_rows_bound(T, k, E)
        self.tq = torch.empty((T, H), dtype=torch.uint8, device=device)
        self.ts = torch.empty((H // 128, T), dtype=torch.float32, device=device)
        self.xq = torch.empty((self.rows, H), dtype=torch.uint8, device=device)
        self.xs = torch.empty((H // 128, self.rows), dtype=torch.float32, device=device)
        # rows outside every segment are never written by the SWIGLU epilogue
        # and stay zero, so their h codes are zero as well
        self.h = torch.zeros((self.rows, F), dtype=torch.bfloat16, device=device)
        self.hq = torch.empty((self.rows, F), dtype=torch.uint8, device=device)
        self.hs = torch.empty((F // 128, self.rows), dtype=torch.float32, device=device)
        self.yrows = torch.empty((self.rows, H), dtype=torch.float32, device=device)
        self.row_of_pair = torch.empty(max(T * k, 1), dtype=torch.int32, device=device)
        self.out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        self._routing_buffers(T, k, device)
        self.disp = None
        from . import load
        wsb = int(load().bs_moe_dispatch_workspace_bytes(T, k, E))
        self.workspace = torch.empty(max(wsb, 16), dtype=torch.uint8, device=device)

    def forward(self, x: torch.Tensor, topk_ids: torch.Tensor, topk_w: torch.Tensor) -> torch.Tensor:
        w = self.w
        self.disp = moe_dispatch(topk_ids, topk_w, w.E, out=self.disp, workspace=self.workspace)
        d = self.disp
        q8_quantize(x, mode=Q8_TOKEN, out=(self.tq, self.ts))
        fp8_gather_rows(self.tq, self.ts, d["token_of"], out=(self.xq, self.xs))
        grouped_gemm_fp8(self.xq, self.xs, w.wgu_codes, w.wgu_sf, N=w.F, E=w.E, offsets=d["offsets"],
                         counts=d["counts"], epilogue=EPI_SWIGLU, out=self.h)
        q8_quantize(self.h, mode=Q8_TOKEN, out=(self.hq, self.hs))
        grouped_gemm_fp8(self.hq, self.hs, w.wd_codes, w.wd_sf, N=w.H, E=w.E, offsets=d["offsets"],
                         counts=d["counts"], epilogue=EPI_ROWS, out=self.yrows, weight_of=d["weight_of"])
        moe_combine(self.yrows, d["pair_of_row"], self.T, self.k, out=self.out, row_of_pair=self.row_of_pair)
        return self.out
