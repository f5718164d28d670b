// gemm_fp4.cu -- persistent warp-specialised block-scaled FP4 GEMM for sm_103a.
//
//   Y = (Q(X) Q(W)^T) (.) scale + L(X) + b
//   ("Warp-specialised W4A4 kernel on the newest GPU architecture", section 1)
//
// One CTA per SM loops over output tiles of 128 x 256 (persistent tile
// scheduling, same page, section 5.3).  Warp roles (section 5.2):
//   warp 0      TMA producer of the main operands: A/B E2M1 codes through
//               128B-swizzled tensor maps, their e4m3 block scales through
//               contiguous bulk copies (the scales are stored in the order the
//               tensor core reads them)
//   warp 1      allocates tensor memory; one lane issues tcgen05.cp (scales
//               shared -> tensor memory) and tcgen05.mma kind::mxf4nvf4 with
//               block16 ue4m3 scales into the fp32 accumulator in tensor
//               memory, then the low-rank MMAs
//   warp 2      TMA producer of the low-rank operands (T hi|lo, Bl^T): its own
//               single-slot pipeline, independent of the main ring
//               (section 4: three independent pipelines)
//   warp 3      builds the grouped tile table, then idles
//   warps 4-11  epilogue: tcgen05.ld of the accumulator (two warps per
//               32-lane quarter, each half of the columns), free the
//               accumulator, then scale / bias / SwiGLU / routed combine and
//               store
// Each role keeps its own PipeState (section 5.1); every wait is bounded.
//
// Grouped mode walks per-expert row segments ("DeepGEMM teardown", 5.3;
// "DeepGEMM for Hopper MoE", 2.2/3): tiles are enumerated expert by expert,
// n-block by n-block, m-block by m-block, from an in-kernel prefix sum of
// ceil(count_e / 128) * n_blocks.
#include "budget.hpp"
#include "kernels.h"
#include "ptx.cuh"

namespace bsk {
namespace fp4 {

constexpr int BM = 128, BN = 256;
constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;
constexpr int kMaxExperts = 1024;
constexpr int kMisc = 2048 + (kMaxExperts + 1) * 4 + 1024;  // barriers + tile table + slack
constexpr int kSfBuffers = 2;
constexpr int kTmemAcc = 0;
constexpr int kTmemSf = BN;                        // scale staging after the accumulator
constexpr int kSfColsPerMma = 4 + BN / 32;         // 4 for A, 8 for B
// Low-rank slot: T hi [128 x 32 bf16], T lo, Bl^T [256 x 32 bf16], 64B swizzle.
constexpr int kLoraThi = 0, kLoraTlo = 8192, kLoraBl = 16384, kLoraBytes = 32768;
constexpr uint32_t kIdescMain = idesc_mxf4nvf4(BM, BN);
constexpr uint32_t kIdescLora = idesc_bf16(BM, BN);

// Stage geometry for a K depth of BK FP4 elements per stage: rows of BK/2
// bytes in the matching TMA / MMA swizzle (128 B for BK = 256, 64 B for 128).
template <int BK>
struct Geo {
  static_assert(BK == 128 || BK == 256, "stage depth");
  static constexpr int kRowBytes = BK / 2;
  static constexpr uint32_t kLayout = BK == 256 ? kLayoutSw128 : kLayoutSw64;
  static constexpr int kSbo = 8 * kRowBytes;              // 8-row swizzle atom
  static constexpr int kMmas = BK / 64;                   // K = 64 per MMA
  static constexpr int kOffA = 0;
  static constexpr int kOffB = BM * kRowBytes;
  static constexpr int kOffSfa = kOffB + BN * kRowBytes;
  static constexpr int kOffSfb = kOffSfa + kMmas * 512;
  static constexpr int kStageBytes = kOffSfb + 2 * kMmas * 512;
  static_assert(kStageBytes % kAlign == 0, "stage alignment");
  static constexpr int kSfColsPerStage = kMmas * kSfColsPerMma;
  static constexpr Fp4TileShape kShapeLora{BM, BN, BK, 1, true, 32, kMisc};
  static constexpr Fp4TileShape kShapeNoLora{BM, BN, BK, 1, false, 32, kMisc};
  static_assert(kStageBytes == fp4_stage_bytes(kShapeNoLora), "stage layout matches the budget");
  static_assert(kLoraBytes == fp4_lora_bytes(kShapeLora), "lora slot layout matches the budget");
  static constexpr int kStagesLora = fp4_main_stages(kShapeLora) < 16 ? fp4_main_stages(kShapeLora) : 16;
  static constexpr int kStagesNoLora = fp4_main_stages(kShapeNoLora) < 16 ? fp4_main_stages(kShapeNoLora) : 16;
  static_assert(kStagesLora >= 2 && kStagesNoLora >= 2, "pipeline needs at least double buffering");
  static_assert(fp4_smem_total(kShapeLora, kStagesLora) + kAlign <= kSmemPerCta, "lora smem");
  static_assert(fp4_smem_total(kShapeNoLora, kStagesNoLora) + kAlign <= kSmemPerCta, "smem");
  static_assert(fp4_tmem_cols(kShapeLora, 1, kSfBuffers) <= kTmemCols, "tmem budget");
  static constexpr int kTmemAlloc = pow2_cols(fp4_tmem_cols(kShapeLora, 1, kSfBuffers));
};

struct Tile {
  int row0;       // first A row (128-aligned)
  int rows;       // valid rows in this tile (<= 128)
  int brow0;      // first B row of accumulator columns [0, 128)
  int brow1;      // first B row of accumulator columns [128, 256)
  int sfb_blk1;   // scale block of brow1 (a valid block even when brow1 is past the weights)
  int col0;       // first output column
  int expert;
};

// Tile fields broadcast from lane 0 (warp-uniform for the issuing roles).
__device__ __forceinline__ Tile bcast_tile(const Tile& t) {
  Tile r;
  r.row0 = warp_bcast(t.row0);
  r.rows = warp_bcast(t.rows);
  r.brow0 = warp_bcast(t.brow0);
  r.brow1 = warp_bcast(t.brow1);
  r.sfb_blk1 = warp_bcast(t.sfb_blk1);
  r.col0 = warp_bcast(t.col0);
  r.expert = warp_bcast(t.expert);
  return r;
}

struct Smem {
  uint8_t* stages;
  uint8_t* lora;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* acc_full;
  uint64_t* acc_empty;
  uint64_t* lora_full;
  uint64_t* lora_empty;
  uint64_t* drain;
  uint32_t* tmem_base;
  int* abort_flag;
  int* total_tiles;
  int* prefix;  // [E + 1]
};

template <int kStages, bool kLora, int kStageBytes>
__device__ __forceinline__ Smem carve(uint8_t* base) {
  Smem s;
  s.stages = base;
  s.lora = base + kStages * kStageBytes;
  uint8_t* misc = s.lora + (kLora ? kLoraBytes : 0);
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
  s.full = bars;
  s.empty = bars + kStages;
  s.acc_full = bars + 2 * kStages;
  s.acc_empty = s.acc_full + 1;
  s.lora_full = s.acc_full + 2;
  s.lora_empty = s.acc_full + 3;
  s.drain = s.acc_full + 4;
  s.tmem_base = reinterpret_cast<uint32_t*>(s.acc_full + 5);
  s.abort_flag = reinterpret_cast<int*>(s.tmem_base + 1);
  s.total_tiles = s.abort_flag + 1;
  s.prefix = s.total_tiles + 2;
  return s;
}

__device__ __forceinline__ int dense_tiles(const Fp4Params& p) {
  return ((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN);
}

template <int kEpi>
__device__ __forceinline__ int n_blocks(const Fp4Params& p) {
  return epi_is_swiglu(kEpi) ? p.N / 128 : (p.N + BN - 1) / BN;
}

template <int kEpi>
__device__ __forceinline__ Tile tile_of(const Fp4Params& p, const int* prefix, int t) {
  Tile tl = {};
  if (p.E == 0) {
    const int num_m = (p.M + BM - 1) / BM;
    const int mb = t % num_m, nb = t / num_m;
    tl.expert = 0;
    tl.row0 = mb * BM;
    tl.rows = min(BM, p.M - tl.row0);
    tl.col0 = nb * BN;
    tl.brow0 = nb * BN;
    tl.brow1 = tl.brow0 + 128;
    tl.sfb_blk1 = (tl.brow1 < p.N) ? tl.brow1 / 128 : tl.brow0 / 128;
    return tl;
  }
  // Grouped: tiles walk chunks of n_chunk column blocks; inside a chunk,
  // expert by expert, column block by column block, row block by row block.
  // prefix[e] = row blocks of experts 0 .. e-1 (prefix[E] = all row blocks).
  const int nbk = n_blocks<kEpi>(p);
  const int nck = (p.n_chunk > 0 && p.n_chunk < nbk) ? p.n_chunk : nbk;
  const int mbt = prefix[p.E];
  const int c = t / (mbt * nck);
  const int nbc = min(nck, nbk - c * nck);
  const int rem = t - c * mbt * nck;
  int lo = 0, hi = p.E - 1;  // largest e with prefix[e] * nbc <= rem
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] * nbc <= rem) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  int eoff, cnt;
  expert_part(p, e, eoff, cnt);
  const int mblk = prefix[e + 1] - prefix[e];
  const int local = rem - prefix[e] * nbc;
  const int nb = c * nck + local / mblk, mb = local % mblk;
  tl.expert = e;
  tl.row0 = eoff + mb * BM;
  tl.rows = min(BM, cnt - mb * BM);
  const int64_t wrows = epi_is_swiglu(kEpi) ? 2LL * p.N : (int64_t)p.N;  // weight rows per expert
  if (epi_is_swiglu(kEpi)) {
    tl.col0 = nb * 128;
    tl.brow0 = (int)(e * wrows + nb * 128);           // gate rows
    tl.brow1 = (int)(e * wrows + p.N + nb * 128);     // up rows
    tl.sfb_blk1 = tl.brow1 / 128;
  } else {
    tl.col0 = nb * BN;
    tl.brow0 = (int)(e * wrows + nb * BN);
    tl.brow1 = tl.brow0 + 128;
    tl.sfb_blk1 = (nb * BN + 128 < p.N) ? tl.brow1 / 128 : tl.brow0 / 128;
  }
  return tl;
}

template <int BK, int kStages, bool kLora, int kEpi>
__global__ void __launch_bounds__(kThreads, 1)
    fp4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmT, const __grid_constant__ CUtensorMap tmL,
                    const Fp4Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + kAlign - 1) &
                                             ~static_cast<uintptr_t>(kAlign - 1));
  using G = Geo<BK>;
  Smem sm = carve<kStages, kLora, G::kStageBytes>(base);
  const int warp = warp_bcast((int)(threadIdx.x / 32)), lane = threadIdx.x % 32;
  volatile int* abort_flag = sm.abort_flag;
  const WaitGuard wg{abort_flag, p.status, p.wait_ns};

  if (threadIdx.x == 0) {
    griddep_launch_dependents();
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(sm.acc_full, 1);
    mbar_init(sm.acc_empty, 8);  // one arrive per epilogue warp
    mbar_init(sm.lora_full, 1);
    mbar_init(sm.lora_empty, 1);
    mbar_init(sm.drain, 1);
    *sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (kLora) {
      prefetch_tmap(&tmT);
      prefetch_tmap(&tmL);
    }
  }
  if (warp == 1) {
    tmem_alloc(sm.tmem_base, G::kTmemAlloc);
    tmem_relinquish();
  }
  // Everything above only touched this CTA's own resources: the operands,
  // expert tables and outputs may belong to the kernel just before this one
  // on the stream (programmatic dependent launch), so wait for it here.
  griddep_wait();
  // alpha times the two-level FP4 tensor scales (powers of two: exact)
  const float alpha_ts = p.alpha * (p.a_ts ? __ldg(p.a_ts) : 1.0f) * (p.b_ts ? __ldg(p.b_ts) : 1.0f);
  if (warp == 3) {
    // Tile table.  Dense: closed form.  Grouped: validate the offset table and
    // prefix-sum the tiles of each expert.
    if (p.E == 0) {
      if (lane == 0) *sm.total_tiles = dense_tiles(p);
    } else {
      const int nb = n_blocks<kEpi>(p);
      int running = 0;
      bool bad = false;
      for (int e0 = 0; e0 < p.E; e0 += 32) {
        const int e = e0 + lane;
        int tiles = 0;
        if (e < p.E) {
          const int off = p.offsets[e], cnt = p.counts[e], nxt = p.offsets[e + 1];
          if (cnt < 0 || (off % BM) != 0 || off + cnt > nxt || nxt > p.M) bad = true;
          int eoff, ecnt;
          expert_part(p, e, eoff, ecnt);
          tiles = (max(ecnt, 0) + BM - 1) / BM;  // row blocks of expert e in this launch
        }
        int incl = tiles;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          int v = __shfl_up_sync(0xffffffffu, incl, d);
          if (lane >= d) incl += v;
        }
        if (e < p.E) sm.prefix[e] = running + incl - tiles;
        running += __shfl_sync(0xffffffffu, incl, 31);
      }
      bad = __any_sync(0xffffffffu, bad) || p.offsets[0] != 0;
      if (lane == 0) {
        sm.prefix[p.E] = running;
        *sm.total_tiles = bad ? 0 : running * nb;
        if (bad && blockIdx.x == 0) record_status(p.status, kStatusOffsets, 1);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = warp_bcast(*sm.tmem_base);
  const int total = warp_bcast(*sm.total_tiles);
  const int kchunks = p.K / 64;
  const int kstages = (kchunks + G::kMmas - 1) / G::kMmas;

  // The three issuing roles below run with the whole warp: lane 0 waits on
  // the barriers (result broadcast), one elected lane issues.
  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    PipeState<kStages> ps;
    uint32_t issued_mask = 0, last_phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile tl = bcast_tile(tile_of<kEpi>(p, sm.prefix, t));
      const uint8_t* sfa_src = p.sfa + (size_t)(tl.row0 / 128) * kchunks * 512;
      const uint8_t* sfb0_src = p.sfb + (size_t)(tl.brow0 / 128) * kchunks * 512;
      const uint8_t* sfb1_src = p.sfb + (size_t)tl.sfb_blk1 * kchunks * 512;
      for (int ks = 0; ks < kstages; ++ks) {
        if (!mbar_wait_warp(&sm.empty[ps.index], ps.phase ^ 1u, wg, 10)) { ok = false; break; }
        const int nmma = min(G::kMmas, kchunks - G::kMmas * ks);
        uint8_t* st = sm.stages + ps.index * G::kStageBytes;
        uint64_t* bar = &sm.full[ps.index];
        if (elect_one()) {
          mbar_arrive_expect_tx(bar, (uint32_t)((BM + BN) * G::kRowBytes + nmma * 512 * 3));
          tma_load_2d(st + G::kOffA, &tmA, bar, ks * G::kRowBytes, tl.row0);
          tma_load_2d(st + G::kOffB, &tmB, bar, ks * G::kRowBytes, tl.brow0);
          tma_load_2d(st + G::kOffB + 128 * G::kRowBytes, &tmB, bar, ks * G::kRowBytes, tl.brow1);
          bulk_load(st + G::kOffSfa, sfa_src + ks * G::kMmas * 512, nmma * 512, bar);
          bulk_load(st + G::kOffSfb, sfb0_src + ks * G::kMmas * 512, nmma * 512, bar);
          bulk_load(st + G::kOffSfb + G::kMmas * 512, sfb1_src + ks * G::kMmas * 512, nmma * 512, bar);
        }
        __syncwarp();
        issued_mask |= 1u << ps.index;
        last_phase = (last_phase & ~(1u << ps.index)) | (ps.phase << ps.index);
        ps.advance();
      }
    }
    if (lane == 0) {
      // Copies already in flight land before the CTA can exit (after an
      // abort; on the normal path every issued stage has completed already).
      for (int s = 0; s < kStages; ++s)
        if (issued_mask & (1u << s)) mbar_drain(&sm.full[s], (last_phase >> s) & 1u, 100000000ull);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------------ low-rank producer
    if (kLora) {
      uint32_t phase = 0;
      bool issued = false;
      for (int t = blockIdx.x; t < total; t += gridDim.x) {
        const Tile tl = bcast_tile(tile_of<kEpi>(p, sm.prefix, t));
        if (!mbar_wait_warp(sm.lora_empty, phase ^ 1u, wg, 20)) break;
        if (elect_one()) {
          mbar_arrive_expect_tx(sm.lora_full, (uint32_t)kLoraBytes);
          tma_load_2d(sm.lora + kLoraThi, &tmT, sm.lora_full, 0, tl.row0);
          tma_load_2d(sm.lora + kLoraTlo, &tmT, sm.lora_full, 32, tl.row0);
          tma_load_2d(sm.lora + kLoraBl, &tmL, sm.lora_full, 0, tl.brow0);
          tma_load_2d(sm.lora + kLoraBl + 8192, &tmL, sm.lora_full, 0, tl.brow1);
        }
        __syncwarp();
        issued = true;
        phase ^= 1u;
      }
      if (issued && lane == 0) mbar_drain(sm.lora_full, phase ^ 1u, 100000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // Per stage: the scale copies (tcgen05.cp, smem -> tensor memory), then the
    // MMAs that read them; both go through the tensor core's in-order stream.
    // Descriptors are built once for stage 0 and advanced by byte offset / 16
    // in their start-address field.
    PipeState<kStages> ps;
    uint32_t acc_phase = 0, lora_phase = 0, sf_buf = 0;
    bool ok = true;
    const uint64_t dA = smem_desc(smem_u32(sm.stages + G::kOffA), 16, G::kSbo, G::kLayout);
    const uint64_t dB = smem_desc(smem_u32(sm.stages + G::kOffB), 16, G::kSbo, G::kLayout);
    const uint64_t dSfa = smem_desc(smem_u32(sm.stages + G::kOffSfa), 0, 128, kLayoutNone);
    const uint64_t dSfb = smem_desc(smem_u32(sm.stages + G::kOffSfb), 0, 128, kLayoutNone);
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      if (!mbar_wait_warp(sm.acc_empty, acc_phase ^ 1u, wg, 30)) break;
      tc_fence_after();
      for (int ks = 0; ks < kstages; ++ks) {
        if (!mbar_wait_warp(&sm.full[ps.index], ps.phase, wg, 31)) { ok = false; break; }
        tc_fence_after();
        const int nmma = min(G::kMmas, kchunks - G::kMmas * ks);
        const uint64_t so = (uint64_t)((ps.index * G::kStageBytes) >> 4);
        const uint32_t sf_col = tmem + kTmemSf + sf_buf * G::kSfColsPerStage;
        if (elect_one()) {
          // each MMA right behind the scale copies it reads (copies and MMAs
          // run in issue order, so the stage's first MMA need not wait for
          // every copy of the stage)
#pragma unroll
          for (int j = 0; j < G::kMmas; ++j) {
            if (j < nmma) {
              const uint32_t col = sf_col + j * kSfColsPerMma;
              tc_cp_32x128b_warpx4(col, dSfa + so + 32 * j);                      // 512 B per block
              tc_cp_32x128b_warpx4(col + 4, dSfb + so + 32 * j);
              tc_cp_32x128b_warpx4(col + 8, dSfb + so + 32 * (G::kMmas + j));
              mma_mxf4nvf4(tmem + kTmemAcc, dA + so + 2 * j, dB + so + 2 * j, kIdescMain, col, col + 4,
                           (ks > 0 || j > 0) ? 1u : 0u);                         // 32 B of K per MMA
            }
          }
          tc_commit(&sm.empty[ps.index]);
        }
        __syncwarp();
        sf_buf ^= 1u;
        ps.advance();
      }
      if (!ok) break;
      if (kLora) {
        if (!mbar_wait_warp(sm.lora_full, lora_phase, wg, 32)) break;
        tc_fence_after();
        if (elect_one()) {
          const uint32_t thi = smem_u32(sm.lora + kLoraThi), tlo = smem_u32(sm.lora + kLoraTlo);
          const uint32_t bl = smem_u32(sm.lora + kLoraBl);
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            const uint32_t ta = part == 0 ? thi : tlo;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
              mma_bf16(tmem + kTmemAcc, smem_desc(ta + 32 * kk, 16, 512, kLayoutSw64),
                       smem_desc(bl + 32 * kk, 16, 512, kLayoutSw64), kIdescLora, 1u);
          }
          tc_commit(sm.lora_empty);
        }
        __syncwarp();
        lora_phase ^= 1u;
      }
      if (elect_one()) tc_commit(sm.acc_full);
      __syncwarp();
      acc_phase ^= 1u;
    }
    // Drain: every tcgen05 op issued above has finished before TMEM is freed.
    if (elect_one()) {
      tc_commit(sm.drain);
      mbar_drain(sm.drain, 0, 1000000000ull);
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp % 4;               // tensor-memory lane quarter
    const int half = (warp - kEpiWarp0) / 4;
    const int r_in_tile = q * 32 + lane;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tl = tile_of<kEpi>(p, sm.prefix, t);
      // one lane polls, the warp follows (keeps the .sync.aligned loads convergent)
      int ok = 1;
      if (lane == 0) ok = mbar_wait(sm.acc_full, acc_phase, wg, 40) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      uint32_t v[4][32];
      const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
      if (epi_is_swiglu(kEpi)) {
        tmem_ld32(lane_base + kTmemAcc + 64 * half, v[0]);
        tmem_ld32(lane_base + kTmemAcc + 64 * half + 32, v[1]);
        tmem_ld32(lane_base + kTmemAcc + 128 + 64 * half, v[2]);
        tmem_ld32(lane_base + kTmemAcc + 128 + 64 * half + 32, v[3]);
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + kTmemAcc + 128 * half + 32 * c, v[c]);
      }
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.acc_empty);
      acc_phase ^= 1u;

      const bool row_ok = r_in_tile < tl.rows;
      const int64_t row = (int64_t)tl.row0 + r_in_tile;
      if (kEpi == kEpiSwiglu && row < p.M) {
        // h = bf16(silu(g) * u); padding rows of the segment are written as zeros.
        const int col = tl.col0 + 64 * half;
        uint16_t* out = reinterpret_cast<uint16_t*>(p.out) + row * p.ldo + col;
#pragma unroll
        for (int c = 0; c < 64; c += 8) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float hv[2];
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
              const int cc = c + 2 * i + k2;
              const float g = __uint_as_float(v[cc / 32][cc % 32]);
              const float u = __uint_as_float(v[2 + cc / 32][cc % 32]);
              hv[k2] = row_ok ? (g / (1.0f + __expf(-g))) * u : 0.0f;
            }
            w[i] = pack_bf16x2(hv[0], hv[1]);
          }
          *reinterpret_cast<uint4*>(out + c) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      } else if (kEpi == kEpiSwigluQ4 && row < p.M) {
        // h quantized in place (see the pair kernel): this warp's 64 columns
        // are one 64-element chunk of h, four groups of 16 on the lane's row;
        // padding rows of the segment get zero codes and scales.
        const int col = tl.col0 + 64 * half;
        uint32_t cw[8];
        uint32_t sfw = 0;
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
          float hx[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = 16 * g4 + i;
            const float g = __uint_as_float(v[c / 32][c % 32]);
            const float u = __uint_as_float(v[2 + c / 32][c % 32]);
            hx[i] = row_ok ? __bfloat162float(__float2bfloat16_rn((g / (1.0f + __expf(-g))) * u)) : 0.0f;
          }
          uint32_t w2[2];
          sfw |= q4_group16_bf16(hx, w2) << (8 * g4);
          cw[2 * g4] = w2[0];
          cw[2 * g4 + 1] = w2[1];
        }
        uint4* dc = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.out) + row * (int64_t)(p.N / 2) + col / 2);
        dc[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
        dc[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
        const int64_t so = ((row / 128) * (int64_t)(p.N / 64) + col / 64) * 512 + (row % 32) * 16 + ((row % 128) / 32) * 4;
        *reinterpret_cast<uint32_t*>(p.out_sf + so) = sfw;
      } else if (kEpi == kEpiCombine) {
        const int col = tl.col0 + 128 * half;
        if (row_ok && row < p.M && col < p.N) {
          const int tok = p.token_of[row];
          const float wt = p.weight_of[row];
          if (tok >= 0) {
            float* dst = p.out32 + (int64_t)tok * p.ld_out32 + col;
#pragma unroll
            for (int c = 0; c < 128; c += 4) {
              const float a0 = wt * __uint_as_float(v[c / 32][c % 32]);
              const float a1 = wt * __uint_as_float(v[c / 32][c % 32 + 1]);
              const float a2 = wt * __uint_as_float(v[c / 32][c % 32 + 2]);
              const float a3 = wt * __uint_as_float(v[c / 32][c % 32 + 3]);
              asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + c), "f"(a0), "f"(a1),
                           "f"(a2), "f"(a3)
                           : "memory");
            }
          }
        }
      } else if (kEpi == kEpiRows) {
        // out[r, n] = weight_of[r] * y[r, n] (fp32) by 32-row groups: a group
        // holding only rows past the expert's count is not written (padding
        // rows of a written group carry weight 0 and become zeros)
        const int col = tl.col0 + 128 * half;
        if (q * 32 < tl.rows && row < p.M && col < p.N) {
          const float wt = p.weight_of[row];
          float* out = reinterpret_cast<float*>(p.out) + row * p.ldo + col;
#pragma unroll
          for (int c = 0; c < 128; c += 4)
            *reinterpret_cast<float4*>(out + c) =
                make_float4(wt * __uint_as_float(v[c / 32][c % 32]), wt * __uint_as_float(v[c / 32][c % 32 + 1]),
                            wt * __uint_as_float(v[c / 32][c % 32 + 2]), wt * __uint_as_float(v[c / 32][c % 32 + 3]));
        }
      } else if (kEpi == kEpiStore) {
        const int col = tl.col0 + 128 * half;
        if (row_ok && row < p.M && col < p.N) {
#pragma unroll
          for (int c = 0; c < 128; c += 8) {
            float y[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int n = col + c + i;
              float a = __uint_as_float(v[(c + i) / 32][(c + i) % 32]);
              float sc = alpha_ts;
              if (p.col_scale) sc *= p.col_scale[n];
              a *= sc;
              if (p.bias) a += __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.bias)[n]);
              y[i] = a;
            }
            if (p.out_bf16) {
              uint16_t* out = reinterpret_cast<uint16_t*>(p.out) + row * p.ldo + col + c;
              *reinterpret_cast<uint4*>(out) = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                                                          pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
            } else {
              float* out = reinterpret_cast<float*>(p.out) + row * p.ldo + col + c;
              *reinterpret_cast<float4*>(out) = make_float4(y[0], y[1], y[2], y[3]);
              *reinterpret_cast<float4*>(out + 4) = make_float4(y[4], y[5], y[6], y[7]);
            }
          }
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, G::kTmemAlloc);
  }
}

template <int BK, bool kLora, int kEpi>
static cudaError_t launch_one(const Fp4Launch& L, cudaStream_t stream) {
  using G = Geo<BK>;
  constexpr int kStages = kLora ? G::kStagesLora : G::kStagesNoLora;
  auto kern = fp4_gemm_kernel<BK, kStages, kLora, kEpi>;
  const int smem = fp4_smem_total(kLora ? G::kShapeLora : G::kShapeNoLora, kStages) + kAlign;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, (unsigned)L.grid, kThreads, (size_t)smem, stream, 1, L.tmA, L.tmB, L.tmT, L.tmL, L.p);
}

template <int BK>
static cudaError_t launch_bk(const Fp4Launch& L, cudaStream_t stream) {
  if (L.lora) {
    if (L.epilogue != kEpiStore) return cudaErrorInvalidValue;
    return launch_one<BK, true, kEpiStore>(L, stream);
  }
  switch (L.epilogue) {
    case kEpiStore: return launch_one<BK, false, kEpiStore>(L, stream);
    case kEpiSwiglu: return launch_one<BK, false, kEpiSwiglu>(L, stream);
    case kEpiSwigluQ4: return launch_one<BK, false, kEpiSwigluQ4>(L, stream);
    case kEpiCombine: return launch_one<BK, false, kEpiCombine>(L, stream);
    case kEpiRows: return launch_one<BK, false, kEpiRows>(L, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fp4

cudaError_t launch_fp4_gemm(const Fp4Launch& L, cudaStream_t stream) {
  if (L.bk == 256) return fp4::launch_bk<256>(L, stream);
  if (L.bk == 128) return fp4::launch_bk<128>(L, stream);
  return cudaErrorInvalidValue;
}

int fp4_stages(bool lora, int bk) {
  if (bk == 256) return lora ? fp4::Geo<256>::kStagesLora : fp4::Geo<256>::kStagesNoLora;
  return lora ? fp4::Geo<128>::kStagesLora : fp4::Geo<128>::kStagesNoLora;
}

}  // namespace bsk
