"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module draws random numbers and nothing else: it holds none of the
quantization, GEMM or MoE arithmetic.  Every array is a deterministic function
of (workload index, shape, seed).  Small arrays come from numpy's PCG64 with
seed 20261202 + workload index; the multi-gigabyte MoE expert weights come
from per-expert torch generators on a chosen device (so a test can regenerate
one expert on its own and copy it to the host).

Workloads (sizes and distributions of the pages' configurations):
  0  dense FP4 tiny:      X[128,512], W[256,512] fp32 ~ N(0,1)
  1  dense FP4 low-rank:  X, W bf16 ~ N(0,1) [8192,8192]; A[K,32], B[32,N]
                          bf16 ~ N(0,0.02); bias[N] bf16 ~ N(0,0.1)
  2  FP8 sweep:           X bf16 [M,4096] ~ N(0,1) with 1% of the channels
                          x50; W bf16 [7168,4096] ~ N(0,0.02)
  3  MoE T=4096 H=4096 E=64 k=8 F=1536
  4  MoE T=16384 H=7168 E=256 k=8 F=2048
  MoE router logits (fp32) ~ N(0,1) + beta_e, beta_e = -1.2 ln(rank_e) for a
  seeded permutation rank of 1..E (log-Zipf, alpha = 1.2).
"""
from __future__ import annotations

import numpy as np
import torch

SEED_BASE = 20261202

DENSE_TINY = dict(M=128, N=256, K=512)
DENSE_LOWRANK = dict(M=8192, N=8192, K=8192, r=32)
FP8_SWEEP = dict(Ms=(1, 16, 64, 128, 4096), N=7168, K=4096)
MOE_SMALL = dict(T=4096, H=4096, E=64, k=8, F=1536)
MOE_LARGE = dict(T=16384, H=7168, E=256, k=8, F=2048)


def rng(index: int, salt: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(SEED_BASE + index + 1000003 * salt))


def normal(g: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    return (g.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def to_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def dense_tiny(M=128, N=256, K=512, index: int = 0):
    g = rng(index)
    return dict(x=torch.from_numpy(normal(g, (M, K))), w=torch.from_numpy(normal(g, (N, K))))


def dense_lowrank(M=8192, N=8192, K=8192, r=32, index: int = 1, lowrank=True, bias=True):
    g = rng(index)
    d = dict(x=to_bf16(normal(g, (M, K))), w=to_bf16(normal(g, (N, K))))
    if lowrank:
        d["lora_a"] = to_bf16(normal(g, (K, r), 0.02))
        d["lora_b"] = to_bf16(normal(g, (r, N), 0.02))
    if bias:
        d["bias"] = to_bf16(normal(g, (N,), 0.1))
    return d


def fp8_sweep(M, N=7168, K=4096, index: int = 2, outlier_frac=0.01, outlier_mult=50.0):
    g = rng(index)
    x = normal(g, (M, K))
    n_out = int(outlier_frac * K)
    ch = g.choice(K, size=n_out, replace=False)
    x[:, ch] *= np.float32(outlier_mult)
    gw = rng(index, salt=1)  # weights independent of M
    w = normal(gw, (N, K), 0.02)
    return dict(x=to_bf16(x), w=to_bf16(w), outlier_channels=np.sort(ch))


def moe_logits(T, E, index: int = 3, zipf_alpha=1.2):
    """Router logits [T, E] fp32: N(0, 1) plus a log-Zipf expert bias
    beta_e = -alpha ln(rank_e) over a seeded permutation rank of 1..E (skewed
    expert loads, some experts empty).  The routing itself (top-k, softmax)
    is part of the path: the GPU router, or the oracle's."""
    g = rng(index, salt=2)
    rank = g.permutation(E) + 1
    beta = -zipf_alpha * np.log(rank.astype(np.float64))
    return (g.standard_normal((T, E)) + beta[None, :]).astype(np.float32)


def moe_activations(T, H, index: int = 3):
    return to_bf16(normal(rng(index, salt=3), (T, H)))


def moe_expert_weights(e: int, F: int, H: int, index: int = 3, device="cpu", std=0.02):
    """Gate/up [2F,H] (gate rows first) and down [H,F] bf16 weights of expert e."""
    gen = torch.Generator(device=device)
    gen.manual_seed(SEED_BASE + index * 100003 + e)
    wgu = (torch.randn((2 * F, H), generator=gen, device=device, dtype=torch.float32) * std)
    wd = (torch.randn((H, F), generator=gen, device=device, dtype=torch.float32) * std)
    return wgu.to(torch.bfloat16), wd.to(torch.bfloat16)
