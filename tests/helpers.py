"""Shared test helpers: the MMA scale layout read back into row-major order
(written from the layout definition in include/bsgemm.h, not from the
library), and the GEMM error bound."""
import numpy as np


def sf_rowmajor(sf, rows, K):
    """MMA-layout e4m3 scale bytes -> [rows, K/16] row-major."""
    sf = np.asarray(sf).reshape(-1)
    G = K // 16
    r = np.arange(rows)[:, None]
    g = np.arange(G)[None, :]
    off = ((r // 128) * (K // 64) + g // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + g % 4
    return sf[off]


def gemm_errors(y, y_ref, S, bf16_out):
    """GEMM tolerance: |y - y_ref| <= 1e-3 * S + 2^-8 |y_ref| (last term bf16 only).
    Returns (ok, max ratio err / bound, max err / S)."""
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_ref)
    bound = 1e-3 * S + (2.0 ** -8 * np.abs(y_ref) if bf16_out else 0.0)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / bound, np.where(err > 0, np.inf, 0.0))
        rel = np.where(S > 0, err / S, 0.0)
    return bool(np.all(err <= bound)), float(ratio.max(initial=0.0)), float(rel.max(initial=0.0))


def tight_errors(y, y_ref, S, bf16_out):
    """A tighter diagnostic bound that fp32 accumulation meets with margin
    (1e-4 S, plus bf16 rounding of the output).  Catches a dropped K group."""
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_ref)
    bound = 1e-4 * S + (2.0 ** -8 * np.abs(y_ref) if bf16_out else 0.0) + 1e-30
    return bool(np.all(err <= bound)), float((err / bound).max(initial=0.0))


def routing(T, E, k, index=3):
    """Seeded router logits and the oracle's top-k routing of them: dict with
    logits fp32 [T, E], topk_ids int32 [T, k], topk_w fp32 [T, k]."""
    import oracle
    import workloads
    logits = workloads.moe_logits(T, E, index=index)
    ids, w = oracle.moe_router(logits, k)
    return dict(logits=logits, topk_ids=ids, topk_w=w.astype(np.float32))
