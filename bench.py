"""Benchmark of the block-scaled GEMM hot path on GB300.

Default workload: dense W4A4 with low-rank branch, M = N = K = 8192, bf16 X and
W ~ N(0,1), A[K,32] and B[32,N] ~ N(0,0.02), bias ~ N(0,0.1), bf16 output.
One step = q4_quantize(X) (codes, scales and the low-rank left factor T = XA)
followed by the block-scaled FP4 GEMM with the low-rank branch and bias; the
weights are quantized once, before timing (they are offline in the method).
Metric: TFLOPS = 2*M*N*K / step time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload dense_lowrank|dense_tiny|fp8_m1|fp8_m16|fp8_m64|fp8_m128|fp8_m4096|moe_small|moe_large]

Under torchrun (N > 1) every rank runs an independent replica of the same
step (the path has no exchange step): value = total work / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

NOMINAL_FP4_OVER_BF16 = 13.5 / 2.25   # dense tensor peaks, profiling recipe table
NOMINAL_FP8_OVER_BF16 = 4.5 / 2.25
NOMINAL_FP4_TFLOPS = 13500.0           # GB300 dense FP4 / FP8 tensor peaks (nominal, per GPU)
NOMINAL_FP8_TFLOPS = 4500.0
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
SPIN_HZ = 2.1e9                        # spin-kernel cycles per second (SM clock, upper bound)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# roofline helpers
# ---------------------------------------------------------------------------
def tensor_roofline(kernel, flops, ms, peaks, source, ratio, nominal_tflops, fmt):
    """Tensor-bound roofline: the FLOPs of one launch over its measured time,
    against the measured bf16 peak times the nominal ratio of `fmt` to bf16,
    with the fraction of the nominal dense peak beside it."""
    tflops = flops / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"] * ratio
    return {"bound": "tensor", "kernel": kernel, "achieved": round(tflops, 1), "peak": round(peak, 1),
            "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
            "peak_source": f"{source} bf16 burst x {ratio:g} (nominal {fmt}/bf16)",
            "nominal": {"peak": nominal_tflops, "frac": round(tflops / nominal_tflops, 4),
                        "source": f"GB300 nominal dense {fmt}"},
            "algorithmic_flops_per_launch": flops, "kernel_ms": round(ms, 5)}


def hbm_roofline(kernel, nbytes, ms, peaks, source):
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak = peaks["hbm_gbs"]
    return {"bound": "hbm", "kernel": kernel, "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
            "frac": round(gbs / peak, 4), "peak_source": f"{source} HBM copy",
            "algorithmic_bytes_per_launch": nbytes, "kernel_ms": round(ms, 5)}


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
class DenseLowRank:
    """Dense W4A4 + low-rank + bias (default), or the tiny fp32 dense case."""

    def __init__(self, tiny=False):
        self.tiny = tiny
        if tiny:
            self.M, self.N, self.K = 128, 256, 512
            self.name = "dense_w4a4_tiny_128x256x512"
        else:
            self.M = self.N = self.K = 8192
            self.name = "dense_w4a4_lowrank_8192x8192x8192_r32_bias_bf16out"
        self.flops = 2.0 * self.M * self.N * self.K
        self.metric = "block-scaled FP4 GEMM TFLOPS (dense W4A4, low-rank branch, bias)"
        self.unit = "TFLOPS"
        self.higher_is_better = True
        self.dtype = "e2m1 x e2m1 (e4m3 group-16 scales), fp32 accumulate, bf16 out"

    def host_inputs(self):
        import workloads
        if self.tiny:
            return workloads.dense_tiny()
        return workloads.dense_lowrank()

    # --- GPU arm
    def setup(self, dev):
        import torch
        import fp8_quantized_gemm_q4_gb300 as bs
        d = self.host_inputs()
        self.h = d
        self.x = d["x"].to(dev)
        w = d["w"].to(dev)
        self.wq, self.ws, _ = bs.q4_quantize(w)
        del w
        M, N, K = self.M, self.N, self.K
        self.xq = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
        self.xs = torch.empty(bs.sf_bytes(M, K), dtype=torch.uint8, device=dev)
        if not self.tiny:
            self.at = d["lora_a"].t().contiguous().to(dev)
            self.bt = d["lora_b"].t().contiguous().to(dev)
            self.bias = d["bias"].to(dev)
            self.lt = torch.empty((M, 64), dtype=torch.bfloat16, device=dev)
            self.out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        else:
            self.at = self.bt = self.bias = self.lt = None
            self.out = torch.empty((M, N), dtype=torch.float32, device=dev)
        self.launches_per_step = 2   # fused quantizer (+ low-rank factor), GEMM
        self.kernel_src = "fp8_quantized_gemm_q4_gb300/csrc/gemm_fp4_pair.cu"
        self.bytes_in = self.x.numel() * self.x.element_size()
        self.bytes_out = self.out.numel() * self.out.element_size()

    def step(self, x=None, gemm_events=None, out=None):
        import fp8_quantized_gemm_q4_gb300 as bs
        x = self.x if x is None else x
        out = self.out if out is None else out
        bs.q4_quantize(x, lora_a_t=self.at, out=(self.xq, self.xs, self.lt))
        if gemm_events:
            gemm_events[0].record()
        bs.gemm_fp4(self.xq, self.xs, self.wq, self.ws, self.K, lora_t=self.lt, lora_b_t=self.bt, bias=self.bias,
                    out=out)
        if gemm_events:
            gemm_events[1].record()
        return out

    def e2e_slots(self, depth):
        """Device buffer sets for the end-to-end pipeline: `depth` copies of
        the activations and of the output (the quantizer's scratch is reused:
        steps run in order on the compute stream)."""
        import torch
        xs = [self.x] + [torch.empty_like(self.x) for _ in range(depth - 1)]
        outs = [self.out] + [torch.empty_like(self.out) for _ in range(depth - 1)]
        return [self.x.cpu().pin_memory()], [[x] for x in xs], outs, lambda s: self.step(xs[s], out=outs[s])

    def roofline(self, gemm_ms, peaks, source):
        return tensor_roofline("fp4_pair_kernel", self.flops, gemm_ms, peaks, source, NOMINAL_FP4_OVER_BF16,
                               NOMINAL_FP4_TFLOPS, "FP4")

    # --- CPU oracle arm
    def oracle_sample(self, rows, cols, nthreads):
        """Quantize `rows` rows of X (+ low-rank factor) and compute their GEMM
        against the first `cols` weight rows with the FP64 oracle."""
        import oracle
        h = self.h
        if not hasattr(self, "_ow"):
            self._ow = {}
        key = cols
        if key not in self._ow:
            self._ow[key] = oracle.q4_quantize(h["w"][:cols])
        ob, osb = self._ow[key]
        x = h["x"][:rows]
        t0 = time.perf_counter()
        oa, osa = oracle.q4_quantize(x)
        t = None if self.tiny else oracle.lowrank_t(x, h["lora_a"])
        oracle.gemm_fp4(oa, osa, ob, osb, self.K, t=t, lora_b=None if self.tiny else h["lora_b"][:, :cols],
                        bias=None if self.tiny else h["bias"][:cols], nthreads=nthreads)
        return time.perf_counter() - t0, 2.0 * rows * cols * self.K


class Fp8Sweep:
    """FP8 e4m3 GEMM, N = 7168, K = 4096, one M of {1, 16, 64, 128, 4096}.
    Step = q8_quantize(X, 1x128) + FP8 GEMM (weights quantized 128x128 once)."""

    def __init__(self, M):
        self.M, self.N, self.K = M, 7168, 4096
        self.name = f"fp8_e4m3_M{M}_N7168_K4096_outliers"
        self.flops = 2.0 * self.M * self.N * self.K
        self.metric = f"FP8 block-scaled GEMM TFLOPS (M={M}, N=7168, K=4096)"
        self.unit = "TFLOPS"
        self.higher_is_better = True
        self.dtype = "e4m3 x e4m3 (fp32 1x128 / 128x128 scales), fp32 accumulate, bf16 out"
        self.kernel_src = "fp8_quantized_gemm_q4_gb300/csrc/gemm_fp8.cu"
        # algorithmic bytes of the GEMM kernel: weights + weight scales + activation codes/scales + output
        self.gemm_bytes = (self.N * self.K + (self.N // 128) * (self.K // 128) * 4 + self.M * self.K
                           + (self.K // 128) * self.M * 4 + self.M * self.N * 2)

    def host_inputs(self):
        import workloads
        return workloads.fp8_sweep(self.M)

    def setup(self, dev):
        import torch
        import fp8_quantized_gemm_q4_gb300 as bs
        d = self.host_inputs()
        self.h = d
        self.x = d["x"].to(dev)
        self.wq, self.ws = bs.q8_quantize(d["w"].to(dev), mode=bs.Q8_BLOCK)
        self.xq = torch.empty((self.M, self.K), dtype=torch.uint8, device=dev)
        self.xs = torch.empty((self.K // 128, self.M), dtype=torch.float32, device=dev)
        self.out = torch.empty((self.M, self.N), dtype=torch.bfloat16, device=dev)
        self.launches_per_step = 2
        self.bytes_in = self.x.numel() * 2
        self.bytes_out = self.out.numel() * 2

    def step(self, x=None, gemm_events=None):
        import fp8_quantized_gemm_q4_gb300 as bs
        x = self.x if x is None else x
        bs.q8_quantize(x, out=(self.xq, self.xs))
        if gemm_events:
            gemm_events[0].record()
        # the weights are quantized once, offline: the GEMM may start loading
        # them while the activation quantizer still runs
        bs.gemm_fp8(self.xq, self.xs, self.wq, self.ws, out=self.out, weights_ready=True)
        if gemm_events:
            gemm_events[1].record()
        return self.out

    def roofline(self, gemm_ms, peaks, source):
        if self.M <= 128:
            return hbm_roofline("fp8_gemm_kernel", self.gemm_bytes, gemm_ms, peaks, source)
        return tensor_roofline("fp8_gemm_kernel", self.flops, gemm_ms, peaks, source, NOMINAL_FP8_OVER_BF16,
                               NOMINAL_FP8_TFLOPS, "FP8")

    def oracle_sample(self, rows, cols, nthreads):
        import oracle
        h = self.h
        if not hasattr(self, "_ow"):
            self._ow = {}
        if cols not in self._ow:
            self._ow[cols] = oracle.q8_quantize(h["w"][:cols], rows_per_block=128)
        ob, osb = self._ow[cols]
        t0 = time.perf_counter()
        oa, osa = oracle.q8_quantize(h["x"][:rows], rows_per_block=1)
        oracle.gemm_fp8(oa, osa, ob, osb, nthreads=nthreads)
        return time.perf_counter() - t0, 2.0 * rows * cols * self.K


class Fp8W8A8(Fp8Sweep):
    """FP8 W8A8 ("Tencent AI Infra interview notes", SmoothQuant): one fp32
    scale per token row of X and per channel of W, Y = s_x[m] s_w[n] sum_k a b
    (no per-block promotion).  Step = q8_quantize(X, per row) + GEMM."""

    def __init__(self, M):
        super().__init__(M)
        self.name = f"fp8_w8a8_M{M}_N7168_K4096_outliers"
        self.metric = f"FP8 W8A8 GEMM TFLOPS (M={M}, N=7168, K=4096, per-token x per-channel scales)"
        self.dtype = "e4m3 x e4m3 (fp32 per-token / per-channel scales), fp32 accumulate, bf16 out"
        self.gemm_bytes = self.N * self.K + self.N * 4 + self.M * self.K + self.M * 4 + self.M * self.N * 2

    def setup(self, dev):
        import torch
        import fp8_quantized_gemm_q4_gb300 as bs
        d = self.host_inputs()
        self.h = d
        self.x = d["x"].to(dev)
        self.wq, self.ws = bs.q8_quantize(d["w"].to(dev), mode=bs.Q8_ROW)
        self.xq = torch.empty((self.M, self.K), dtype=torch.uint8, device=dev)
        self.xs = torch.empty((self.M,), dtype=torch.float32, device=dev)
        self.out = torch.empty((self.M, self.N), dtype=torch.bfloat16, device=dev)
        self.launches_per_step = 2
        self.bytes_in = self.x.numel() * 2
        self.bytes_out = self.out.numel() * 2

    def step(self, x=None, gemm_events=None):
        import fp8_quantized_gemm_q4_gb300 as bs
        x = self.x if x is None else x
        bs.q8_quantize(x, mode=bs.Q8_ROW, out=(self.xq, self.xs))
        if gemm_events:
            gemm_events[0].record()
        bs.gemm_fp8(self.xq, self.xs, self.wq, self.ws, out=self.out, weights_ready=True, rowwise=True)
        if gemm_events:
            gemm_events[1].record()
        return self.out

    def oracle_sample(self, rows, cols, nthreads):
        import oracle
        h = self.h
        if not hasattr(self, "_ow"):
            self._ow = {}
        if cols not in self._ow:
            self._ow[cols] = oracle.q8_quantize_rowwise(h["w"][:cols])
        ob, osb = self._ow[cols]
        t0 = time.perf_counter()
        oa, osa = oracle.q8_quantize_rowwise(h["x"][:rows])
        oracle.gemm_fp8_rowwise(oa, osa, ob, osb)
        return time.perf_counter() - t0, 2.0 * rows * cols * self.K


class Fp4Decode(Fp8Sweep):
    """Dense W4A4 decode: M tokens (<= 32) against N = 7168, K = 4096 FP4
    weights ("Tencent AI Infra interview notes", decode intensity: 2KN FLOPs
    per KN/2 weight bytes).  X bf16 N(0, 1) with the FP8 sweep's outlier
    channels, W N(0, 0.02).  Step = q4_quantize(X) + the decode GEMM."""

    def __init__(self, M):
        super().__init__(M)
        self.name = f"fp4_decode_M{M}_N7168_K4096"
        self.metric = f"FP4 decode GEMM TFLOPS (M={M}, N=7168, K=4096)"
        self.dtype = "e2m1 x e2m1 (e4m3 group-16 scales), fp32 accumulate, bf16 out"
        self.kernel_src = "fp8_quantized_gemm_q4_gb300/csrc/gemm_fp4_decode.cu"
        N, K, M = self.N, self.K, self.M
        self.gemm_bytes = N * K // 2 + N * K // 16 + M * K // 2 + 128 * K // 16 + M * N * 2

    def setup(self, dev):
        import torch
        import fp8_quantized_gemm_q4_gb300 as bs
        d = self.host_inputs()
        self.h = d
        self.x = d["x"].to(dev)
        self.wq, self.ws, _ = bs.q4_quantize(d["w"].to(dev))
        self.xq = torch.empty((self.M, self.K // 2), dtype=torch.uint8, device=dev)
        self.xs = torch.empty(bs.sf_bytes(self.M, self.K), dtype=torch.uint8, device=dev)
        self.out = torch.empty((self.M, self.N), dtype=torch.bfloat16, device=dev)
        self.launches_per_step = 2
        self.bytes_in = self.x.numel() * 2
        self.bytes_out = self.out.numel() * 2

    def step(self, x=None, gemm_events=None):
        import fp8_quantized_gemm_q4_gb300 as bs
        x = self.x if x is None else x
        bs.q4_quantize(x, out=(self.xq, self.xs, None))
        if gemm_events:
            gemm_events[0].record()
        bs.gemm_fp4(self.xq, self.xs, self.wq, self.ws, self.K, out=self.out, weights_ready=True)
        if gemm_events:
            gemm_events[1].record()
        return self.out

    def roofline(self, gemm_ms, peaks, source):
        return hbm_roofline("fp4_decode_kernel", self.gemm_bytes, gemm_ms, peaks, source)

    def oracle_sample(self, rows, cols, nthreads):
        import oracle
        h = self.h
        if not hasattr(self, "_ow"):
            self._ow = {}
        if cols not in self._ow:
            self._ow[cols] = oracle.q4_quantize(h["w"][:cols])
        ob, osb = self._ow[cols]
        t0 = time.perf_counter()
        oa, osa = oracle.q4_quantize(h["x"][:rows])
        oracle.gemm_fp4(oa, osa, ob, osb, self.K, nthreads=nthreads)
        return time.perf_counter() - t0, 2.0 * rows * cols * self.K


class DecodeChain(Fp8Sweep):
    """Decode GEMMs back to back: one activation quantization of M = 16 tokens,
    then G = 8 GEMMs of [16 x 4096] by different [7168 x 4096] weight sets (as
    the projections of a decode step that read the same activation), each a
    programmatic dependent launch with weights_ready, so its weight stream
    starts under the tail of the GEMM before it.  fmt "fp8": block-scaled FP8
    (swap-AB stream-K kernel); "fp4": the FP4 decode kernel.  multi: the same
    G products as one bs_gemm_multi launch (one tile list on one grid);
    otherwise the G GEMMs replay as one captured CUDA graph behind the eager
    quantizer.
    Roofline: the G GEMMs' algorithmic bytes over the time from the first
    GEMM's start to the last one's end (the quantizer excluded)."""

    G = 8

    def __init__(self, fmt, multi=False):
        super().__init__(16)
        self.fmt = fmt
        self.multi = multi  # the G products in one bs_gemm_multi launch
        G = self.G
        if multi:
            self.name = f"{fmt}_decode_multi_{G}x_M16_N7168_K4096"
            self.metric = f"{fmt.upper()} decode multi-weight GEMM TFLOPS ({G} weight sets in one launch, " \
                          f"M=16, N=7168, K=4096)"
        else:
            self.name = f"{fmt}_decode_chain_{G}x_M16_N7168_K4096"
            self.metric = f"{fmt.upper()} decode GEMM chain TFLOPS ({G} GEMMs, M=16, N=7168, K=4096)"
        self.flops = G * 2.0 * self.M * self.N * self.K
        N, K, M = self.N, self.K, self.M
        if fmt == "fp4":
            self.dtype = "e2m1 x e2m1 (e4m3 group-16 scales), fp32 accumulate, bf16 out"
            self.kernel_src = "fp8_quantized_gemm_q4_gb300/csrc/gemm_fp4_decode.cu"
            one = N * K // 2 + N * K // 16 + M * K // 2 + 128 * K // 16 + M * N * 2
        else:
            one = self.gemm_bytes
        self.gemm_bytes = G * one

    def setup(self, dev):
        import torch
        import fp8_quantized_gemm_q4_gb300 as bs
        import workloads
        d = self.host_inputs()
        self.h = d
        self.x = d["x"].to(dev)
        M, N, K = self.M, self.N, self.K
        self.ws_list = []
        for g in range(self.G):
            gen = torch.Generator(device=dev)
            gen.manual_seed(workloads.SEED_BASE + 7919 * (g + 1))
            w = (torch.randn(N, K, generator=gen, device=dev) * 0.02).to(torch.bfloat16)
            if self.fmt == "fp4":
                wq, wsf, _ = bs.q4_quantize(w)
            else:
                wq, wsf = bs.q8_quantize(w, mode=bs.Q8_BLOCK)
            self.ws_list.append((wq, wsf))
            del w
        if self.fmt == "fp4":
            self.xq = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
            self.xs = torch.empty(bs.sf_bytes(M, K), dtype=torch.uint8, device=dev)
        else:
            self.xq = torch.empty((M, K), dtype=torch.uint8, device=dev)
            self.xs = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
        self.outs = torch.empty((self.G, M, N), dtype=torch.bfloat16, device=dev)
        self.out_list = [self.outs[g] for g in range(self.G)]
        self.out = self.outs[-1]
        self.launches_per_step = 2 if self.multi else 1 + self.G
        self.bytes_in = self.x.numel() * 2
        self.bytes_out = self.out.numel() * 2
        self.graph = None
        if not self.multi:
            self._capture_gemms()

    def _gemms(self):
        import fp8_quantized_gemm_q4_gb300 as bs
        for g, (wq, wsf) in enumerate(self.ws_list):
            if self.fmt == "fp4":
                bs.gemm_fp4(self.xq, self.xs, wq, wsf, self.K, out=self.outs[g], weights_ready=True)
            else:
                bs.gemm_fp8(self.xq, self.xs, wq, wsf, out=self.outs[g], weights_ready=True)

    def _capture_gemms(self):
        """The G chained GEMMs as one CUDA graph (their programmatic-dependent
        launches kept as graph edges), so that a step costs the host two
        launches (quantizer, graph) instead of 1 + G library calls, and the
        timed steps measure the device rather than the host's enqueue rate.
        The stream-K workspace of the capture stream exists before capture
        (a warm-up call on that stream allocates it)."""
        import torch
        import fp8_quantized_gemm_q4_gb300 as bs
        if self.fmt == "fp4":
            bs.q4_quantize(self.x, out=(self.xq, self.xs, None))
        else:
            bs.q8_quantize(self.x, out=(self.xq, self.xs))
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self._gemms()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                self._gemms()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.graph = g

    def step(self, x=None, gemm_events=None):
        import fp8_quantized_gemm_q4_gb300 as bs
        x = self.x if x is None else x
        if self.fmt == "fp4":
            bs.q4_quantize(x, out=(self.xq, self.xs, None))
        else:
            bs.q8_quantize(x, out=(self.xq, self.xs))
        if gemm_events:
            gemm_events[0].record()
        if self.multi:
            if self.fmt == "fp4":
                bs.gemm_fp4_multi(self.xq, self.xs, self.ws_list, self.K, outs=self.out_list, weights_ready=True)
            else:
                bs.gemm_fp8_multi(self.xq, self.xs, self.ws_list, outs=self.out_list, weights_ready=True)
            if gemm_events:
                gemm_events[1].record()
            return self.out
        if self.graph is not None:
            self.graph.replay()
        else:
            self._gemms()
        if gemm_events:
            gemm_events[1].record()
        return self.out

    def roofline(self, gemm_ms, peaks, source):
        if self.multi:
            kern = ("fp4_decode_kernel" if self.fmt == "fp4" else "fp8_gemm_kernel") + \
                f" (multi-weight: {self.G} products, one launch)"
        else:
            kern = ("fp4_decode_kernel" if self.fmt == "fp4" else "fp8_gemm_kernel") + f" x{self.G} (chain)"
        return hbm_roofline(kern, self.gemm_bytes, gemm_ms, peaks, source)


class DenseTwoLevel(DenseLowRank):
    """Dense W4A4 8192^3 with two-level FP4 operands (power-of-two tensor
    scale above the e4m3 group scales; weights N(0, 0.02)), bf16 out, no
    low-rank branch.  Step = tensor amax + two-level quantize of X + GEMM."""

    def __init__(self):
        super().__init__(tiny=False)
        self.name = "dense_w4a4_two_level_8192x8192x8192_bf16out"
        self.metric = "block-scaled FP4 GEMM TFLOPS (dense W4A4, two-level scales)"
        self.dtype = "e2m1 x e2m1 (e4m3 group-16 x power-of-two tensor scales), fp32 accumulate, bf16 out"

    def host_inputs(self):
        import workloads
        d = workloads.dense_lowrank(lowrank=False, bias=False)
        d["w"] = (d["w"].float() * 0.02).to(d["w"].dtype)
        return d

    def setup(self, dev):
        import torch
        import fp8_quantized_gemm_q4_gb300 as bs
        d = self.host_inputs()
        self.h = d
        self.x = d["x"].to(dev)
        self.wq, self.ws, self.wts = bs.q4_quantize_two_level(d["w"].to(dev))
        M, N, K = self.M, self.N, self.K
        self.xq = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
        self.xs = torch.empty(bs.sf_bytes(M, K), dtype=torch.uint8, device=dev)
        self.xts = torch.empty(1, dtype=torch.float32, device=dev)
        self.amax = torch.empty(1, dtype=torch.float32, device=dev)
        self.out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        self.launches_per_step = 4   # amax (zero + reduce), quantize, GEMM
        self.kernel_src = "fp8_quantized_gemm_q4_gb300/csrc/gemm_fp4_pair.cu"
        self.bytes_in = self.x.numel() * 2
        self.bytes_out = self.out.numel() * 2

    def step(self, x=None, gemm_events=None):
        import fp8_quantized_gemm_q4_gb300 as bs
        x = self.x if x is None else x
        bs.tensor_amax(x, out=self.amax)
        bs.q4_quantize_two_level(x, amax=self.amax, out=(self.xq, self.xs, self.xts))
        if gemm_events:
            gemm_events[0].record()
        bs.gemm_fp4(self.xq, self.xs, self.wq, self.ws, self.K, out=self.out, a_tensor_scale=self.xts,
                    b_tensor_scale=self.wts)
        if gemm_events:
            gemm_events[1].record()
        return self.out

    def oracle_sample(self, rows, cols, nthreads):
        import oracle
        h = self.h
        if not hasattr(self, "_ow"):
            self._ow = {}
        if cols not in self._ow:
            self._ow[cols] = oracle.q4_quantize_two_level(h["w"][:cols])
        ob, osb, tb = self._ow[cols]
        t0 = time.perf_counter()
        oa, osa, ta = oracle.q4_quantize_two_level(h["x"][:rows])
        oracle.gemm_fp4(oa, osa, ob, osb, self.K, alpha=ta * tb, nthreads=nthreads)
        return time.perf_counter() - t0, 2.0 * rows * cols * self.K


class MoEWorkload:
    """Grouped FP4 MoE layer from router logits: top-k router, dispatch, quantize +
    gather, gate/up GEMM + SwiGLU with h re-quantized, down GEMM, routed combine
    (one step = one layer)."""

    def __init__(self, large, combine="rows", graph=True, h_quant="fused"):
        import workloads
        self.combine = combine
        self.h_quant = h_quant
        self.graph = graph  # the layer replayed as one CUDA graph
        cfg = workloads.MOE_LARGE if large else workloads.MOE_SMALL
        self.index = 4 if large else 3
        self.T, self.H, self.E, self.k, self.F = cfg["T"], cfg["H"], cfg["E"], cfg["k"], cfg["F"]
        self.M, self.N, self.K = self.T, self.H, self.H
        self.name = f"moe_fp4_T{self.T}_H{self.H}_E{self.E}_k{self.k}_F{self.F}"
        self.metric = f"MoE grouped FP4 layer TFLOPS (T={self.T}, H={self.H}, E={self.E}, k={self.k}, F={self.F})"
        self.unit = "TFLOPS"
        self.higher_is_better = True
        self.dtype = "e2m1 x e2m1 (e4m3 group-16 scales), fp32 accumulate, bf16 out"
        # real rows only: gate/up 2*rows*H*2F, down 2*rows*F*H
        rows = self.T * self.k
        self.flops = 2.0 * rows * self.H * 2 * self.F + 2.0 * rows * self.F * self.H

    def host_inputs(self):
        import workloads
        return dict(x=workloads.moe_activations(self.T, self.H, index=self.index),
                    logits=workloads.moe_logits(self.T, self.E, index=self.index))

    def setup(self, dev):
        import torch
        import workloads
        from fp8_quantized_gemm_q4_gb300.moe import MoELayer, quantize_expert_weights
        d = self.host_inputs()
        self.h = d
        self.x = d["x"].to(dev)
        self.logits = torch.from_numpy(d["logits"]).to(dev)
        gu, dn = [], []
        W = None
        # quantize expert by expert so the bf16 weights never all sit on the device
        import fp8_quantized_gemm_q4_gb300 as bs
        F2, H, F, E = 2 * self.F, self.H, self.F, self.E
        wgu_codes = torch.empty((E * F2, H // 2), dtype=torch.uint8, device=dev)
        wgu_sf = torch.empty(bs.sf_bytes(E * F2, H), dtype=torch.uint8, device=dev)
        wd_codes = torch.empty((E * H, F // 2), dtype=torch.uint8, device=dev)
        wd_sf = torch.empty(bs.sf_bytes(E * H, F), dtype=torch.uint8, device=dev)
        pg, pd = bs.sf_bytes(F2, H), bs.sf_bytes(H, F)
        for e in range(E):
            wgu, wd = workloads.moe_expert_weights(e, F, H, index=self.index, device=dev)
            bs.q4_quantize(wgu, out=(wgu_codes[e * F2:(e + 1) * F2], wgu_sf[e * pg:(e + 1) * pg], None))
            bs.q4_quantize(wd, out=(wd_codes[e * H:(e + 1) * H], wd_sf[e * pd:(e + 1) * pd], None))
        from fp8_quantized_gemm_q4_gb300.moe import MoEWeights
        W = MoEWeights(E, H, F, wgu_codes, wgu_sf, wd_codes, wd_sf)
        self.layer = MoELayer(W, self.T, self.k, device=dev, combine=self.combine, h_quant=self.h_quant)
        self.out = self.layer.out
        if self.graph:
            # capture once (router included); from here on the workload's
            # inputs are the graph's static ones
            self.layer.capture(self.x, logits=self.logits)
            self.x, self.logits = self.layer.static_x, self.layer.static_logits
        # router 1 + dispatch 3 + quantize 1 + gather 1 + gate/up GEMM (+ quantize
        # h 1 on the separate path) + down GEMM, then combine 3 (invert, init,
        # sum) or finalize 2 (cast, zero); each grouped GEMM is two launches on
        # CTA pairs with the small experts split off (the library's default)
        g = 2   # CTA pairs plus the one-CTA launch for experts of <= 128 rows (the library's default)
        self.launches_per_step = 1 + (5 if self.layer.h_quant == "fused" else 6) + 2 * g + \
            (3 if self.combine == "rows" else 2)
        self.bytes_in = self.x.numel() * 2 + self.logits.numel() * 4
        self.bytes_out = self.out.numel() * 2
        # expert loads of this routing, from the layer's own router output
        self.layer.replay() if self.graph else self.layer.forward_logits(self.x, self.logits)
        counts = torch.bincount(self.layer.topk_ids.flatten().long(), minlength=E).cpu()
        self.load_hist = {"max": int(counts.max()), "min": int(counts.min()), "empty": int((counts == 0).sum())}

    def e2e_buffers(self):
        import torch
        return [(self.x.cpu().pin_memory(), self.x if self.graph else torch.empty_like(self.x)),
                (self.logits.cpu().pin_memory(), self.logits)]

    def step(self, x=None, gemm_events=None):
        x = self.x if x is None else x
        if gemm_events:
            gemm_events[0].record()
        if self.graph:
            # the graph reads the static inputs (self.x / logits are those)
            out = self.layer.replay(None if x is self.x else x)
        else:
            out = self.layer.forward_logits(x, self.logits)
        if gemm_events:
            gemm_events[1].record()
        return out

    def algorithmic_bytes(self):
        """Bytes the layer must move at least: every expert's FP4 weights and
        their scales (read once), the bf16 activations and fp32 router logits
        in, the bf16 output."""
        E, H, F, T = self.E, self.H, self.F, self.T
        w = E * (2 * F * H + H * F)
        return w // 2 + w // 16 + T * H * 2 + T * E * 4 + T * H * 2

    def roofline(self, layer_ms, peaks, source):
        kern = ("whole layer (grouped fp4_pair_kernel x2 + quantize + dispatch + " +
                ("combine" if self.combine == "rows" else "finalize") + ")")
        r = tensor_roofline(kern, self.flops, layer_ms, peaks, source, NOMINAL_FP4_OVER_BF16, NOMINAL_FP4_TFLOPS,
                            "FP4")
        h = hbm_roofline(kern, self.algorithmic_bytes(), layer_ms, peaks, source)
        r["hbm"] = {k: h[k] for k in ("achieved", "peak", "unit", "frac", "peak_source",
                                      "algorithmic_bytes_per_launch")}
        r["expert_load"] = getattr(self, "load_hist", None)
        return r

    def oracle_sample(self, rows, cols, nthreads):
        """`rows` tokens through the oracle's layer (cols ignored)."""
        import oracle
        import workloads
        h = self.h
        t0 = time.perf_counter()
        ids, wts = oracle.moe_router(h["logits"][:rows], self.k)
        t_router = time.perf_counter() - t0
        toks = list(range(rows))
        experts = sorted(set(int(e) for t in toks for e in ids[t]))
        if not hasattr(self, "_ow"):
            self._ow = {}
        for e in experts:
            if e not in self._ow:
                wgu, wd = workloads.moe_expert_weights(e, self.F, self.H, index=self.index, device="cuda")
                self._ow[e] = (oracle.q4_quantize(wgu.cpu()), oracle.q4_quantize(wd.cpu()))
        E = self.E
        gc = [self._ow[e][0][0] if e in self._ow else None for e in range(E)]
        gs = [self._ow[e][0][1] if e in self._ow else None for e in range(E)]
        dc = [self._ow[e][1][0] if e in self._ow else None for e in range(E)]
        ds = [self._ow[e][1][1] if e in self._ow else None for e in range(E)]
        t0 = time.perf_counter()
        oracle.moe_layer(h["x"][:rows], ids, wts.astype("float32"), gc, gs, dc, ds, F=self.F, nthreads=nthreads)
        fl = 2.0 * rows * self.k * (self.H * 2 * self.F + self.F * self.H)
        return time.perf_counter() - t0 + t_router, fl


class QuantWorkload:
    """Activation quantizer alone, an HBM-bound kernel: "q4" = FP4 (E2M1 codes,
    e4m3 group-16 scales) of the 8192 x 8192 bf16 activations of the dense
    workload; "q8" = FP8 1x128 token blocks of the 4096 x 4096 bf16
    activations of the FP8 prefill workload.  value = algorithmic bytes per
    second (TB/s; the bytes take the place of FLOPs in the common fields)."""

    def __init__(self, kind):
        self.kind = kind
        if kind == "q4":
            self.M = self.K = 8192
            self.name = "q4_quantize_bf16_8192x8192"
            self.metric = "FP4 activation quantizer HBM throughput (8192 x 8192 bf16)"
            per_elem = 2 + 0.5 + 1 / 16
            self.kernel = "q4_quantize_kernel"
        else:
            self.M, self.K = 4096, 4096
            self.name = "q8_quantize_token_bf16_4096x4096_outliers"
            self.metric = "FP8 1x128 token quantizer HBM throughput (4096 x 4096 bf16)"
            per_elem = 2 + 1 + 4 / 128
            self.kernel = "q8_token_kernel"
        self.N = self.K
        self.flops = per_elem * self.M * self.K   # algorithmic bytes
        self.unit = "TB/s"
        self.higher_is_better = True
        self.dtype = "bf16 in; e2m1 codes + e4m3 scales out" if kind == "q4" else "bf16 in; e4m3 codes + fp32 scales out"
        self.launches_per_step = 1

    def host_inputs(self):
        import workloads
        return workloads.dense_lowrank() if self.kind == "q4" else workloads.fp8_sweep(4096)

    def setup(self, dev):
        import torch
        import fp8_quantized_gemm_q4_gb300 as bs
        d = self.host_inputs()
        self.h = d
        self.x = d["x"].to(dev)
        M, K = self.M, self.K
        if self.kind == "q4":
            self.outs = (torch.empty((M, K // 2), dtype=torch.uint8, device=dev),
                         torch.empty(bs.sf_bytes(M, K), dtype=torch.uint8, device=dev), None)
        else:
            self.outs = (torch.empty((M, K), dtype=torch.uint8, device=dev),
                         torch.empty((K // 128, M), dtype=torch.float32, device=dev))
        self.out = self.outs[0]   # the codes: what the end-to-end pass reads back
        self.bytes_in = self.x.numel() * 2
        self.bytes_out = self.out.numel()

    def step(self, x=None, gemm_events=None):
        import fp8_quantized_gemm_q4_gb300 as bs
        x = self.x if x is None else x
        if gemm_events:
            gemm_events[0].record()
        if self.kind == "q4":
            bs.q4_quantize(x, out=self.outs)
        else:
            bs.q8_quantize(x, out=self.outs)
        if gemm_events:
            gemm_events[1].record()
        return self.out

    def roofline(self, kern_ms, peaks, source):
        return hbm_roofline(self.kernel, self.flops, kern_ms, peaks, source)

    def oracle_sample(self, rows, cols, nthreads):
        import oracle
        x = self.h["x"][:rows]
        t0 = time.perf_counter()
        if self.kind == "q4":
            oracle.q4_quantize(x)
        else:
            oracle.q8_quantize(x, 1)
        return time.perf_counter() - t0, self.flops * rows / self.M


class Fp8MoEWorkload(MoEWorkload):
    """Grouped FP8 MoE layer from router logits (e4m3 with fp32 scales per 1x128
    token block and 128x128 expert weight block): router, dispatch, quantize +
    gather, gate/up GEMM with the SwiGLU epilogue, h quantize, down GEMM with
    weighted rows, routed combine (one step = one layer, one CUDA graph)."""

    def __init__(self, large=False):
        super().__init__(large)
        self.name = f"moe_fp8_T{self.T}_H{self.H}_E{self.E}_k{self.k}_F{self.F}"
        self.metric = f"MoE grouped FP8 layer TFLOPS (T={self.T}, H={self.H}, E={self.E}, k={self.k}, F={self.F})"
        self.dtype = "e4m3 x e4m3 (fp32 1x128 / 128x128 block scales), fp32 accumulate, bf16 out"

    def setup(self, dev):
        import torch
        import workloads
        from fp8_quantized_gemm_q4_gb300.moe import Fp8MoELayer, Fp8MoEWeights
        import fp8_quantized_gemm_q4_gb300 as bs
        d = self.host_inputs()
        self.h = d
        self.x = d["x"].to(dev)
        self.logits = torch.from_numpy(d["logits"]).to(dev)
        F2, H, F, E = 2 * self.F, self.H, self.F, self.E
        wgu_codes = torch.empty((E * F2, H), dtype=torch.uint8, device=dev)
        wgu_sf = torch.empty((E * F2 // 128, H // 128), dtype=torch.float32, device=dev)
        wd_codes = torch.empty((E * H, F), dtype=torch.uint8, device=dev)
        wd_sf = torch.empty((E * H // 128, F // 128), dtype=torch.float32, device=dev)
        bg, bd = F2 // 128, H // 128
        # quantize expert by expert so the bf16 weights never all sit on the device
        for e in range(E):
            wgu, wd = workloads.moe_expert_weights(e, F, H, index=self.index, device=dev)
            bs.q8_quantize(wgu, mode=bs.Q8_BLOCK, out=(wgu_codes[e * F2:(e + 1) * F2], wgu_sf[e * bg:(e + 1) * bg]))
            bs.q8_quantize(wd, mode=bs.Q8_BLOCK, out=(wd_codes[e * H:(e + 1) * H], wd_sf[e * bd:(e + 1) * bd]))
        W = Fp8MoEWeights(E, H, F, wgu_codes, wgu_sf, wd_codes, wd_sf)
        self.layer = Fp8MoELayer(W, self.T, self.k, device=dev)
        self.out = self.layer.out
        self.layer.capture(self.x, logits=self.logits)
        self.x, self.logits = self.layer.static_x, self.layer.static_logits
        # router 1 + dispatch 3 + quantize 1 + gather 1 + gate/up GEMM 1 +
        # quantize h 1 + down GEMM 1 + combine 3
        self.launches_per_step = 12
        self.bytes_in = self.x.numel() * 2 + self.logits.numel() * 4
        self.bytes_out = self.out.numel() * 2
        self.layer.replay()
        counts = torch.bincount(self.layer.topk_ids.flatten().long(), minlength=E).cpu()
        self.load_hist = {"max": int(counts.max()), "min": int(counts.min()), "empty": int((counts == 0).sum())}

    def algorithmic_bytes(self):
        """Every expert's FP8 weights and their 128x128 block scales (read
        once), the bf16 activations and fp32 router logits in, the bf16 output."""
        E, H, F, T = self.E, self.H, self.F, self.T
        w = E * (2 * F * H + H * F)
        return w + (w // (128 * 128)) * 4 + T * H * 2 + T * E * 4 + T * H * 2

    def roofline(self, layer_ms, peaks, source):
        kern = "whole layer (fp8_grouped_kernel x2 + quantize x2 + gather + router + dispatch + combine)"
        r = tensor_roofline(kern, self.flops, layer_ms, peaks, source, NOMINAL_FP8_OVER_BF16, NOMINAL_FP8_TFLOPS,
                            "FP8")
        h = hbm_roofline(kern, self.algorithmic_bytes(), layer_ms, peaks, source)
        r["hbm"] = {k: h[k] for k in ("achieved", "peak", "unit", "frac", "peak_source",
                                      "algorithmic_bytes_per_launch")}
        r["expert_load"] = getattr(self, "load_hist", None)
        return r

    def oracle_sample(self, rows, cols, nthreads):
        """`rows` tokens through the oracle's FP8 layer (cols ignored)."""
        import oracle
        import workloads
        h = self.h
        t0 = time.perf_counter()
        ids, wts = oracle.moe_router(h["logits"][:rows], self.k)
        t_router = time.perf_counter() - t0
        experts = sorted(set(int(e) for t in range(rows) for e in ids[t]))
        if not hasattr(self, "_ow8"):
            self._ow8 = {}
        for e in experts:
            if e not in self._ow8:
                wgu, wd = workloads.moe_expert_weights(e, self.F, self.H, index=self.index, device="cuda")
                self._ow8[e] = (oracle.q8_quantize(wgu.cpu(), 128), oracle.q8_quantize(wd.cpu(), 128))
        E = self.E
        pick = lambda i, j: [self._ow8[e][i][j] if e in self._ow8 else None for e in range(E)]
        t0 = time.perf_counter()
        oracle.moe_layer(h["x"][:rows], ids, wts.astype("float32"), pick(0, 0), pick(0, 1), pick(1, 0), pick(1, 1),
                         F=self.F, nthreads=nthreads, fmt="fp8")
        fl = 2.0 * rows * self.k * (self.H * 2 * self.F + self.F * self.H)
        return time.perf_counter() - t0 + t_router, fl


WORKLOADS = {
    "dense_lowrank": lambda: DenseLowRank(tiny=False),
    "dense_tiny": lambda: DenseLowRank(tiny=True),
    "fp8_m1": lambda: Fp8Sweep(1),
    "fp8_m16": lambda: Fp8Sweep(16),
    "fp8_m64": lambda: Fp8Sweep(64),
    "fp8_m128": lambda: Fp8Sweep(128),
    "fp8_m4096": lambda: Fp8Sweep(4096),
    "fp8_w8a8_m16": lambda: Fp8W8A8(16),
    "fp8_w8a8_m4096": lambda: Fp8W8A8(4096),
    "dense_two_level": lambda: DenseTwoLevel(),
    "fp4_decode_m1": lambda: Fp4Decode(1),
    "fp4_decode_m16": lambda: Fp4Decode(16),
    "moe_small": lambda: MoEWorkload(large=False),
    "moe_large": lambda: MoEWorkload(large=True),
    "moe_fp8_small": lambda: Fp8MoEWorkload(large=False),
    "fp8_decode_chain": lambda: DecodeChain("fp8"),
    "fp8_decode_multi": lambda: DecodeChain("fp8", multi=True),
    "fp4_decode_multi": lambda: DecodeChain("fp4", multi=True),
    "fp4_decode_chain": lambda: DecodeChain("fp4"),
    "q4_quantize": lambda: QuantWorkload("q4"),
    "q8_quantize": lambda: QuantWorkload("q8"),
}


KERNEL_HEADERS = ("budget.hpp", "kernels.h", "ptx.cuh")


def _code_only(path: str) -> bytes:
    """Source text without comments or blank lines (comment edits do not
    change the kernel a profile was taken on)."""
    import re
    text = open(path, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip()).encode()


def kernel_source_sha1(kernel_src: str) -> str:
    """sha1 over the code of a kernel's translation unit followed by the shared
    device headers it includes (in KERNEL_HEADERS order), comments removed: a
    change to either makes a recorded profile stale."""
    h = hashlib.sha1(_code_only(os.path.join(ROOT, kernel_src)))
    csrc = os.path.dirname(os.path.join(ROOT, kernel_src))
    for name in KERNEL_HEADERS:
        h.update(_code_only(os.path.join(csrc, name)))
    return h.hexdigest()


def traffic_for(kernel_src: str, workload: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel source (and headers) and
    this workload (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    h = kernel_source_sha1(kernel_src)
    for ent in d.get("entries", []):
        if ent.get("kernel_src") == kernel_src and ent.get("source_sha1") == h and ent.get("workload") == workload:
            return ent.get("dram_bytes_per_launch")
    return None


# ---------------------------------------------------------------------------
def max_over_ranks(values, device):
    """Element-wise max of per-rank timings (the slowest replica sets the job's
    time).  Works with NCCL on GPUs and gloo on CPU."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(work_per_rank, world, step_ms):
    """Whole-job rate: all ranks' work over the (max-over-ranks) step time."""
    return world * work_per_rank / (step_ms * 1e-3)


def time_steps(args, wl, world, dev):
    """W untimed warm-up steps, then two timed passes of K steps, each step
    bracketed by CUDA events on the launching stream (L2 flushed before every
    step, outside the events), with the GPU clocks sampled during both:
      - the step pass records no event inside a step, so a kernel may start
        under the tail of the one before it (programmatic dependent launch)
        exactly as in use: its times give ms_per_step;
      - the kernel pass also records events around the dominant kernel (which
        serialises it against its neighbours): its times give the kernel's
        own duration for the roofline.
    Returns (step ms, dominant-kernel ms, clocks, wall seconds), the times
    max-over-ranks."""
    import torch
    import torch.distributed as dist
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    clean = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def flush_l2(i):
        # Write a buffer larger than L2, then read another one: the step's
        # operands are evicted, and what L2 holds afterwards is clean, so the
        # timed kernels do not pay for writing back the flush's dirty lines.
        flush.fill_(float(i))
        clean.sum()

    for i in range(args.warmup):
        flush_l2(i)
        wl.step()
    torch.cuda.synchronize()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[torch.cuda.current_device()]))
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    wall0 = time.perf_counter()
    for events, kernel_events in ((ev, None), (kev, gev)):
        # Hold the stream with a spin kernel while the host enqueues the K
        # steps, so that the steps then run back to back: the events time the
        # GPU's work, not gaps in which the device waited for host-side
        # launches (binding and tensor-map set-up take tens of microseconds
        # per call, as long as a whole decode step).  The end-to-end figure
        # keeps them.
        torch.cuda._sleep(int((K * 400e-6 + 5e-3) * SPIN_HZ))
        for i in range(K):
            flush_l2(i)                    # L2 flush, outside the per-step events
            events[i][0].record(stream)
            wl.step(gemm_events=None if kernel_events is None else kernel_events[i])
            events[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    del flush, clean
    step_ms = sum(a.elapsed_time(b) for a, b in ev) / K
    gemm_ms = sum(a.elapsed_time(b) for a, b in gev) / K
    step_ms, gemm_ms = max_over_ranks([step_ms, gemm_ms], dev)
    return step_ms, gemm_ms, clk, wall


def check_device_status():
    import fp8_quantized_gemm_q4_gb300 as bs
    st, detail = bs.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({detail:#x}) after the timed region")


# The other configurations of the metric ("block-scaled FP4/FP8 GEMM TFLOPS &
# % of GB300 dense peak; MoE layer us"), timed in the same run as the dense
# headline and reported beside it.
EXTRAS = ("moe_small", "moe_large", "moe_fp8_small", "fp8_m16", "fp8_m4096", "fp8_w8a8_m16", "fp8_w8a8_m4096",
          "fp4_decode_m16", "fp8_decode_chain", "fp8_decode_multi", "fp4_decode_chain", "fp4_decode_multi", "q4_quantize", "q8_quantize")


def run_extra(args, name, world, dev, peaks, source):
    import torch
    wl = WORKLOADS[name]()
    wl.setup(dev)
    step_ms, kern_ms, clk, wall = time_steps(args, wl, world, dev)
    check_device_status()
    roof = wl.roofline(kern_ms, peaks, source)
    roof["traffic"] = traffic_for(wl.kernel_src, wl.name) if hasattr(wl, "kernel_src") else None
    d = {"metric": wl.metric, "value": round(job_throughput(wl.flops, world, step_ms) / 1e12, 2), "unit": wl.unit,
         "workload": wl.name, "ms_per_step": round(step_ms, 5), "us_per_step": round(step_ms * 1e3, 2),
         "kernel_ms": round(kern_ms, 5), "gpu_launches": 2 * args.steps * wl.launches_per_step,
         "roofline": roof, "clocks": clk, "timed_wall_s": round(wall, 3)}
    del wl
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return d


def run_ours(args, wl, rank, world, dev, peaks, source):
    import torch
    wl.setup(dev)
    stream = torch.cuda.current_stream()
    K = args.steps
    step_ms, gemm_ms, clk, wall = time_steps(args, wl, world, dev)

    # End to end through the public API with pinned host buffers: every step
    # copies all its inputs host -> device and its result device -> host.
    # CopyComputePipeline overlaps the copies in, the step and the copies out
    # of consecutive steps on three streams (workloads with e2e_slots get two
    # buffer sets; others one, so their copies overlap the neighbouring steps'
    # copies only).  Workloads with several inputs name them as (host,
    # device) pairs, the first being the activations.
    from fp8_quantized_gemm_q4_gb300.pipeline import CopyComputePipeline
    if hasattr(wl, "e2e_slots"):
        hosts, din, dout, stepf = wl.e2e_slots(2)
    else:
        pairs = wl.e2e_buffers() if hasattr(wl, "e2e_buffers") else [(wl.x.cpu().pin_memory(), torch.empty_like(wl.x))]
        hosts, din, dout = [h for h, _ in pairs], [[d for _, d in pairs]], [wl.out]
        stepf = lambda s: wl.step(din[0][0])
    yh = torch.empty(dout[0].shape, dtype=dout[0].dtype).pin_memory()
    pipe = CopyComputePipeline(stepf, din, dout)
    Ke = args.e2e_steps if args.e2e_steps > 0 else max(1, min(K, 100))
    for _ in range(3):
        pipe.submit(hosts, yh)
    pipe.finish()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(Ke):
        pipe.submit(hosts, yh)
    pipe.finish()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / Ke
    (e2e_ms,) = max_over_ranks([e2e_ms], dev)
    e2e_overlap = (f"copies in / step / copies out of consecutive steps on three streams, {len(dout)} device "
                   "buffer set(s)")

    check_device_status()
    value = job_throughput(wl.flops, world, step_ms) / 1e12
    roof = wl.roofline(gemm_ms, peaks, source)
    roof["traffic"] = traffic_for(getattr(wl, "kernel_src", "fp8_quantized_gemm_q4_gb300/csrc/gemm_fp4.cu"),
                                  wl.name)
    line = {
        "metric": wl.metric, "value": round(value, 2), "unit": wl.unit, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": wl.higher_is_better,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic (seeded, pages' shapes)",
        "config": {"workload": wl.name, "M": wl.M, "N": wl.N, "K": wl.K,
                   "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write, then {L2_FLUSH_BYTES >> 20} MiB "
                         "read so L2 holds clean lines; outside the step events)",
                   "enqueue": "timed steps queued behind a GPU spin (device time without host launch gaps)",
                   "parallelism": f"replicas x{world}",
                   **({"moe_combine": wl.combine, "cuda_graph": wl.graph,
                       "h_quant": getattr(wl.layer, "h_quant", "separate")}
                      if hasattr(wl, "combine") else {})},
        "e2e": {"value": round(job_throughput(wl.flops, world, e2e_ms) / 1e12, 2), "unit": wl.unit,
                "ms_per_step": round(e2e_ms, 5), "overlap": e2e_overlap, "h2d_bytes_per_step": wl.bytes_in,
                "d2h_bytes_per_step": wl.bytes_out},
        "gpu_launches": 2 * K * wl.launches_per_step,   # two timed passes
        "roofline": roof,
        "clocks": clk,
        "timed_wall_s": round(wall, 3),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_seconds)
    if args.workload == "dense_lowrank" and not args.no_extras:
        h = getattr(wl, "h", None)
        del wl, h
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        line["extra"] = {name: run_extra(args, name, world, dev, peaks, source) for name in EXTRAS}
    return line


def cpu_baseline(wl, budget_s=15.0):
    """The FP64 oracle timed on the host cores on a bounded sample of rows
    (threads split rows, so the sample is a multiple of the thread count)."""
    import oracle
    oracle.build()
    nthreads = oracle.default_threads()
    cols = wl.N
    dt1, _ = wl.oracle_sample(1, cols, 1)                  # calibration: one row, one thread
    rows = min(wl.M, max(1, int(budget_s / max(dt1, 1e-6))) * nthreads)
    dt, fl = wl.oracle_sample(rows, cols, nthreads)
    return {"value": round(fl / dt / 1e12, 8), "unit": wl.unit, "cores": min(nthreads, rows), "kind": "oracle",
            "sample": f"{rows} rows x {cols} cols x K={wl.K} (quantize + low-rank + GEMM), {dt:.1f} s",
            "seconds": round(dt, 2)}


def run_reference(args, wl):
    """The oracle as the reference arm: each step one bounded sample of the
    workload (one row per host thread against a slice of the columns)."""
    import oracle
    oracle.build()
    wl.h = wl.host_inputs()
    nthreads = oracle.default_threads()
    rows = min(wl.M, nthreads)
    dt1, _ = wl.oracle_sample(1, wl.N, 1)                  # one row, one thread, all columns
    total_steps = args.steps + args.warmup
    per_step = max(0.01, 90.0 / max(total_steps, 1))
    cols = max(128, min(wl.N, int(wl.N * per_step / max(dt1, 1e-6)) // 128 * 128))
    for _ in range(args.warmup):
        wl.oracle_sample(rows, cols, nthreads)
    tot_t = tot_f = 0.0
    for _ in range(args.steps):
        t, f = wl.oracle_sample(rows, cols, nthreads)
        tot_t += t
        tot_f += f
    value = tot_f / tot_t / 1e12
    sample = f"{rows} rows x {cols} cols x K={wl.K} per step (quantize + low-rank + GEMM)"
    return {
        "impl": "reference", "metric": wl.metric, "value": round(value, 8), "unit": wl.unit, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_t / args.steps * 1e3, 3),
        "higher_is_better": wl.higher_is_better, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 (oracle)", "data": "synthetic (seeded, pages' shapes)",
        "config": {"workload": wl.name, "M": wl.M, "N": wl.N, "K": wl.K, "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 8), "unit": wl.unit, "cores": rows, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 8), "unit": wl.unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="dense_lowrank", choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="dense headline only (by default the MoE layers and the FP8 M=16 / M=4096 shapes are "
                         "timed in the same run and reported under 'extra')")
    ap.add_argument("--e2e-steps", type=int, default=0, help="end-to-end steps (default min(steps, 100))")
    ap.add_argument("--moe-combine", choices=["rows", "atomic"], default="rows",
                    help="MoE routed combine: weighted rows + per-token sum, or fp32 reductions")
    ap.add_argument("--moe-h-quant", choices=["fused", "separate"], default="fused",
                    help="MoE: quantize h in the gate/up epilogue (default) or in a separate pass")
    ap.add_argument("--moe-eager", action="store_true",
                    help="MoE: launch the layer's kernels one by one instead of replaying its CUDA graph")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    wl = WORKLOADS[args.workload]()
    if isinstance(wl, MoEWorkload):
        wl.combine = args.moe_combine
        wl.graph = not args.moe_eager
        wl.h_quant = args.moe_h_quant

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, wl)), flush=True)
        return

    import torch
    import torch.distributed as dist
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    import __graft_entry__
    __graft_entry__.build()
    peaks, source = load_peaks()
    line = run_ours(args, wl, rank, world, dev, peaks, source)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
