// budget.hpp -- build-time shared-memory / tensor-memory budget of the
// block-scaled GEMM kernels.
//
// "Warp-specialised W4A4 kernel on the newest GPU architecture", section 6:
// the kernel solves a shared-memory budget at build time,
//     smem_total = main_stages * (bytes_A + bytes_B) + lora_stages * bytes_lora + misc
//     smem_total <= SMEM per SM,
// maximising main_stages first and lora_stages second; its bug was counting
// the per-CTA low-rank up-projection block twice in 2-CTA mode (each CTA of
// a pair holds only its half), which silently drove main_stages to the
// minimum.  Every byte term here states whether it is split across the CTAs
// of a pair or replicated in each, and the kernels static_assert the result.
//
// Plain C++17 constexpr, no CUDA dependence, so host unit tests can include it.
#pragma once
#include <stdint.h>

namespace bsk {

constexpr int kSmemPerCta = 232448;  // 227 KiB opt-in dynamic shared memory per CTA (sm_100 family)
constexpr int kTmemCols = 512;       // tensor-memory columns per SM (128 lanes x 32 bit)
constexpr int kAlign = 1024;         // 128B-swizzle atoms repeat every 1024 bytes

constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }

struct Fp4TileShape {
  int BM;         // rows of A per CTA (MMA M per CTA)
  int BN;         // columns of the pair's MMA (N); each CTA of a pair holds BN / cta_pair rows of B
  int BK;         // K elements per pipeline stage
  int cta_pair;   // 1 or 2 CTAs cooperating on one MMA
  bool lora;      // low-rank branch present
  int lora_r;     // rank of the low-rank branch
  int misc;       // barriers, tile tables and alignment slack
};

// Bytes of one main-pipeline stage held by ONE CTA.
//   A codes:   BM x BK/2                        (own rows, never shared)
//   B codes:   (BN / cta_pair) x BK/2           (split: each CTA of a pair loads half of B)
//   A scales:  BM x BK/16                       (own rows)
//   B scales:  BN x BK/16                       (replicated: the MMA of either CTA reads all BN scale rows)
constexpr int fp4_stage_bytes(Fp4TileShape s) {
  return s.BM * s.BK / 2 + (s.BN / s.cta_pair) * s.BK / 2 + s.BM * s.BK / 16 + s.BN * s.BK / 16;
}

// Bytes of one low-rank stage held by ONE CTA: T hi|lo rows of its own M
// block (bf16, 2r wide) plus its share of the up-projection block Bl^T
// (bf16, BN x r) -- split across a pair, NOT replicated.
constexpr int fp4_lora_bytes(Fp4TileShape s) {
  return s.lora ? (s.BM * 2 * s.lora_r * 2 + (s.BN / s.cta_pair) * s.lora_r * 2) : 0;
}

// The accounting bug of the page, kept only so the unit tests can show what
// it costs: the up-projection block counted in full by every CTA of a pair.
constexpr int fp4_lora_bytes_replicated(Fp4TileShape s) {
  return s.lora ? (s.BM * 2 * s.lora_r * 2 + s.BN * s.lora_r * 2) : 0;
}

constexpr int fp4_lora_stages(Fp4TileShape s) { return s.lora ? 1 : 0; }

// Largest main_stages that fits next to the low-rank stages and misc bytes.
constexpr int max_main_stages(int stage_bytes, int lora_total, int misc, int limit = kSmemPerCta) {
  return (limit - lora_total - misc) / stage_bytes;
}

constexpr int fp4_main_stages(Fp4TileShape s) {
  return max_main_stages(round_up(fp4_stage_bytes(s), kAlign),
                         fp4_lora_stages(s) * round_up(fp4_lora_bytes(s), kAlign), s.misc);
}

constexpr int fp4_smem_total(Fp4TileShape s, int stages) {
  return stages * round_up(fp4_stage_bytes(s), kAlign) + fp4_lora_stages(s) * round_up(fp4_lora_bytes(s), kAlign) +
         s.misc;
}

// Tensor-memory columns: one fp32 accumulator of BN columns (128 lanes = BM
// rows), plus block-scale staging for `sf_buffers` stages of BK / 64 MMAs,
// each needing 4 columns for A scales and BN / 32 columns for B scales.
constexpr int fp4_tmem_cols(Fp4TileShape s, int acc_buffers, int sf_buffers) {
  return acc_buffers * s.BN + sf_buffers * (s.BK / 64) * (4 + s.BN / 32);
}

constexpr int pow2_cols(int c) { return c <= 32 ? 32 : c <= 64 ? 64 : c <= 128 ? 128 : c <= 256 ? 256 : 512; }

// ---- FP8 (kind::f8f6f4) tiles: fp32 scales are applied per 128-K block by
// the epilogue warps, so the tensor memory holds `partial_buffers` per-block
// partial accumulators of BN columns each.
struct Fp8TileShape {
  int BM, BN, BK;  // BK == 128: one scale block per stage
  int misc;
};
constexpr int fp8_stage_bytes(Fp8TileShape s) { return s.BM * s.BK + s.BN * s.BK; }
constexpr int fp8_main_stages(Fp8TileShape s) {
  return max_main_stages(round_up(fp8_stage_bytes(s), kAlign), 0, s.misc);
}
constexpr int fp8_smem_total(Fp8TileShape s, int stages) {
  return stages * round_up(fp8_stage_bytes(s), kAlign) + s.misc;
}

}  // namespace bsk
