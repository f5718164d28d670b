// gemm_fp4_pair.cu -- block-scaled FP4 GEMM on CTA pairs (tcgen05 cta_group::2).
//
// "Warp-specialised W4A4 kernel on the newest GPU architecture", sections 4-6:
// two CTAs form a pair that shares one 256 x 256 MMA; switching the MMA mode
// alone gains nothing (section 4, 27 % -> 28 %): the data and sync flows are
// split per CTA, and the shared-memory budget counts per CTA what each CTA
// actually holds (section 6: the up-projection block of the low-rank branch
// is split across the pair, not replicated).
//
// Per CTA of a pair (cluster of 2), per K stage of 128 FP4 elements (the
// default 256-element stage holds twice each):
//   A      its own 128 rows                     8 KB  (64B swizzle)
//   B      its own half (128 rows) of the 256   8 KB
//   SFA    scales of its own rows               1 KB
//   SFB    scales of all 256 B rows             2 KB  (held by both: each CTA's
//          tensor core multiplies its rows by all 256 columns, so each CTA
//          loads both 128-row blocks itself)
// so a 128-deep stage is 19 KB instead of 27 KB, and 10-11 stages fit.
//
// The leader CTA (rank 0) issues every tcgen05.mma / tcgen05.cp with
// cta_group::2; the operands of the peer live at the same shared-memory
// offsets in the peer.  Both CTAs' TMA loads signal the leader's "full"
// barrier (the leader expects the bytes of both); the leader's commits
// multicast to both CTAs' "empty" / "acc_full" barriers; both CTAs' epilogue
// warps arrive on the leader's "acc_empty".  Each CTA's tensor memory holds
// the fp32 accumulator of its own 128 rows x 256 columns.
#include "budget.hpp"
#include "kernels.h"
#include "ptx.cuh"

namespace bsk {
namespace fp4pair {

constexpr int BM = 128;        // rows per CTA (the pair covers 256)
constexpr int BN = 256;        // MMA N; each CTA holds BN / 2 rows of B
constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;
constexpr int kMaxExperts = 1024;
constexpr int kMiscBase = 2048 + 1024;                 // barriers, tile count + slack
constexpr int kMiscTable = (kMaxExperts + 1) * 4;     // expert row-block prefix table (grouped only)
// Output staging for TMA stores: one buffer per epilogue warp holding a box
// of 32 rows.  Without the low-rank branch a box row is 64 bytes (32 bf16 or
// 16 fp32 columns) in the 64-byte swizzle layout (16-byte chunk j of row r at
// j ^ ((r >> 1) & 3)); the low-rank variant, short of shared memory, uses
// 32-byte rows in the 32-byte swizzle layout (chunk j at j ^ ((r >> 2) & 1)).
// Either way the lanes' 16-byte writes fall in distinct banks.
template <bool kLora>
struct EpiBox {
  static constexpr int kRowW = kLora ? 8 : 16;     // 32-bit words per box row
  static constexpr int kRowBytes = 4 * kRowW;
  static constexpr int kBytes = 32 * kRowBytes;    // per warp
  static constexpr int kStage = 8 * kBytes;        // 8 epilogue warps
};
constexpr int kEpiStageLora = EpiBox<true>::kStage;
constexpr int kEpiStageNoLora = EpiBox<false>::kStage;
// low-rank slot per CTA: T hi / T lo of its own rows, its half of Bl^T
constexpr int kLoraThi = 0, kLoraTlo = 8192, kLoraBl = 16384, kLoraBytes = 24576;
constexpr int kSfBuffers = 2;
constexpr int kTmemAcc = 0;
constexpr int kTmemSf = BN;
constexpr int kSfColsPerMma = 4 + BN / 32;

// Per-CTA stage geometry for a K depth of BK FP4 elements per stage.
template <int BK>
struct PGeo {
  static_assert(BK == 128 || BK == 256, "stage depth");
  static constexpr int kRowBytes = BK / 2;
  static constexpr uint32_t kLayout = BK == 256 ? kLayoutSw128 : kLayoutSw64;
  static constexpr int kSbo = 8 * kRowBytes;
  static constexpr int kMmas = BK / 64;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = BM * kRowBytes;
  static constexpr int kOffSfa = kOffB + (BN / 2) * kRowBytes;
  static constexpr int kOffSfb = kOffSfa + kMmas * 512;
  static constexpr int kStageBytes = kOffSfb + 2 * kMmas * 512;
  static constexpr int kStageTx = kStageBytes;  // bytes one CTA's loads deliver per stage
  static constexpr int kSfWords = kMmas * 128;  // scale words of one 128-row block per stage
  static constexpr int kSfBox = kSfWords / 2;     // one TMA box per stage: BK 8-byte elements
  // the low-rank branch is dense-only, so its variant carries no expert table
  static constexpr Fp4TileShape kShapeLora{BM, BN, BK, 2, true, 32, kMiscBase + kEpiStageLora};
  static constexpr Fp4TileShape kShapeNoLora{BM, BN, BK, 2, false, 32, kMiscBase + kMiscTable + kEpiStageNoLora};
  static_assert(kStageBytes == fp4_stage_bytes(kShapeNoLora), "per-CTA stage layout matches the budget");
  static_assert(kStageBytes % kAlign == 0, "stage alignment");
  static_assert(kLoraBytes == fp4_lora_bytes(kShapeLora), "low-rank slot: the up-projection block is split per CTA");
  static constexpr int kStagesLora = fp4_main_stages(kShapeLora) < 16 ? fp4_main_stages(kShapeLora) : 16;
  static constexpr int kStagesNoLora = fp4_main_stages(kShapeNoLora) < 16 ? fp4_main_stages(kShapeNoLora) : 16;
  static_assert(fp4_smem_total(kShapeLora, kStagesLora) + kAlign <= kSmemPerCta, "lora smem");
  static_assert(fp4_smem_total(kShapeNoLora, kStagesNoLora) + kAlign <= kSmemPerCta, "smem");
  static constexpr int kSfColsPerStage = kMmas * kSfColsPerMma;
  static_assert(fp4_tmem_cols(kShapeLora, 1, kSfBuffers) <= kTmemCols, "tmem budget");
  static constexpr int kTmemAlloc = pow2_cols(fp4_tmem_cols(kShapeLora, 1, kSfBuffers));
};

constexpr uint32_t kIdescMain = idesc_mxf4nvf4(2 * BM, BN);
constexpr uint32_t kIdescLora = idesc_bf16(2 * BM, BN);
// half tiles (256 x 128) of the dense tail, see dense_work()
constexpr uint32_t kIdescMainHalf = idesc_mxf4nvf4(2 * BM, BN / 2);
constexpr uint32_t kIdescLoraHalf = idesc_bf16(2 * BM, BN / 2);

struct Tile {
  int row0;      // first A row of the pair (this CTA's rows start at row0 + rank * 128)
  int rows;      // valid rows of the pair tile (<= 256)
  int brow0;     // first B row of accumulator columns [0, 128)   (leader's half)
  int brow1;     // first B row of accumulator columns [128, 256) (peer's half)
  int sfb_blk1;  // scale block of brow1 (valid even when brow1 is past the weights)
  int col0;      // first output column
  int narrow;    // 1: a 256 x 128 half tile (MMA N = 128, accumulator columns [0, 128))
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
  r.narrow = warp_bcast(t.narrow);
  return r;
}

template <int kEpi>
__device__ __forceinline__ int n_blocks(const Fp4Params& p) {
  return epi_is_swiglu(kEpi) ? p.N / 128 : (p.N + BN - 1) / BN;
}

// Dense work list.  With T pair tiles on P pairs, the last T mod P tiles
// would run as a partial wave while the other pairs idle (8192^3: 1024 tiles
// on 76 pairs, 36 pairs doing 14 tiles and 40 doing 13).  When that tail
// fits in half the pairs, each tail tile is split into two 256 x 128 halves
// (MMA N = 128) so that the tail spreads over twice as many pairs.
// Returns the number of work items; `full` receives the count of whole tiles.
// Only the plain dense epilogue (kEpiStore) splits.
template <int kEpi>
__device__ __forceinline__ int dense_work(const Fp4Params& p, int npairs, int& full) {
  const int tiles = ((p.M + 2 * BM - 1) / (2 * BM)) * ((p.N + BN - 1) / BN);
  const int tail = tiles % npairs;
  full = tiles;
  if (kEpi != kEpiStore || !p.half_tail || tail == 0 || 2 * tail > npairs) return tiles;
  full = tiles - tail;
  return tiles + tail;
}

template <int kEpi>
__device__ __forceinline__ Tile tile_of(const Fp4Params& p, const int* prefix, int t) {
  Tile tl = {};
  if (p.E == 0) {
    int nfull;
    dense_work<kEpi>(p, (int)(gridDim.x / 2), nfull);
    int half = -1;
    if (t >= nfull) {  // half tile: item nfull + 2 i + h is half h of tile nfull + i
      half = (t - nfull) & 1;
      t = nfull + (t - nfull) / 2;
    }
    const int num_m = (p.M + 2 * BM - 1) / (2 * BM);
    const int mb = t % num_m, nb = t / num_m;
    tl.row0 = mb * 2 * BM;
    tl.rows = min(2 * BM, p.M - tl.row0);
    if (half < 0) {
      tl.col0 = nb * BN;
      tl.brow0 = nb * BN;
      tl.brow1 = tl.brow0 + 128;
      tl.sfb_blk1 = (tl.brow1 < p.N) ? tl.brow1 / 128 : tl.brow0 / 128;
    } else {
      // each CTA supplies 64 of the 128 B rows at its B offset: the leader
      // rows [brow0, brow0 + 64), the peer [brow0 + 64, brow0 + 128); the
      // other 64 rows of each CTA's 128-row box are loaded but not used
      tl.narrow = 1;
      tl.col0 = nb * BN + 128 * half;
      tl.brow0 = tl.col0;
      tl.brow1 = tl.brow0 + 64;
      tl.sfb_blk1 = tl.brow0 / 128;
    }
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
  tl.row0 = eoff + mb * 2 * BM;
  tl.rows = min(2 * BM, cnt - mb * 2 * BM);
  const int64_t wrows = epi_is_swiglu(kEpi) ? 2LL * p.N : (int64_t)p.N;
  if (epi_is_swiglu(kEpi)) {
    tl.col0 = nb * 128;
    tl.brow0 = (int)(e * wrows + nb * 128);
    tl.brow1 = (int)(e * wrows + p.N + nb * 128);
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
    fp4_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmT, const __grid_constant__ CUtensorMap tmL,
                    const __grid_constant__ CUtensorMap tmSfa, const __grid_constant__ CUtensorMap tmSfb,
                    const __grid_constant__ CUtensorMap tmO, const Fp4Params p) {
  using G = PGeo<BK>;
  constexpr int kStageBytes = G::kStageBytes, kRowBytes = G::kRowBytes, kMmas = G::kMmas;
  constexpr int kOffA = G::kOffA, kOffB = G::kOffB, kOffSfa = G::kOffSfa, kOffSfb = G::kOffSfb;
  constexpr int kSbo = G::kSbo, kSfColsPerStage = G::kSfColsPerStage, kTmemAlloc = G::kTmemAlloc;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + kAlign - 1) &
                                             ~static_cast<uintptr_t>(kAlign - 1));
  uint8_t* stages = base;
  uint8_t* lora = base + kStages * kStageBytes;
  using Box = EpiBox<kLora>;
  uint8_t* estage = lora + (kLora ? kLoraBytes : 0);  // [8 warps][Box::kBytes]
  uint64_t* bars = reinterpret_cast<uint64_t*>(estage + Box::kStage);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* acc_full = bars + 2 * kStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* lora_full = acc_full + 2;
  uint64_t* lora_empty = acc_full + 3;
  uint64_t* drain = acc_full + 4;
  uint32_t* tmem_base = reinterpret_cast<uint32_t*>(acc_full + 5);
  int* abort_i = reinterpret_cast<int*>(tmem_base + 1);
  int* total_tiles = abort_i + 1;
  int* prefix = total_tiles + 2;
  volatile int* abort_flag = abort_i;
  const WaitGuard wg{abort_flag, p.status, p.wait_ns};

  const int warp = warp_bcast((int)(threadIdx.x / 32)), lane = threadIdx.x % 32;
  const uint32_t rank = warp_bcast(cluster_ctarank());
  const bool leader = rank == 0;
  const int pair = blockIdx.x / 2, npairs = gridDim.x / 2;

  if (threadIdx.x == 0) {
    griddep_launch_dependents();
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 16);  // 8 epilogue warps in each CTA of the pair
    mbar_init(lora_full, 1);
    mbar_init(lora_empty, 1);
    mbar_init(drain, 1);
    *abort_i = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmSfa);
    prefetch_tmap(&tmSfb);
    if (kEpi == kEpiSwiglu || kEpi == kEpiRows || (kEpi == kEpiStore && p.E == 0)) prefetch_tmap(&tmO);
    if (kLora) {
      prefetch_tmap(&tmT);
      prefetch_tmap(&tmL);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_base, kTmemAlloc);
    tmem_relinquish_pair();
  }
  // Everything above only touched this CTA's own resources: the operands,
  // expert tables and outputs may belong to the kernel just before this one
  // on the stream (programmatic dependent launch), so wait for it here.
  griddep_wait();
  // alpha times the two-level FP4 tensor scales (powers of two: exact)
  const float alpha_ts = p.alpha * (p.a_ts ? __ldg(p.a_ts) : 1.0f) * (p.b_ts ? __ldg(p.b_ts) : 1.0f);
  if (warp == 3) {
    if (p.E == 0) {
      int nfull;
      const int items = dense_work<kEpi>(p, npairs, nfull);
      if (lane == 0) *total_tiles = items;
    } else if (kLora) {
      // the low-rank variant has no expert table: nothing to do (the host never asks for this)
      if (lane == 0) {
        *total_tiles = 0;
        if (blockIdx.x == 0) record_status(p.status, kStatusOffsets, 4);
      }
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
          tiles = (max(ecnt, 0) + 2 * BM - 1) / (2 * BM);  // row blocks (pairs) of expert e in this launch
        }
        int incl = tiles;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, d);
          if (lane >= d) incl += v;
        }
        if (e < p.E) prefix[e] = running + incl - tiles;
        running += __shfl_sync(0xffffffffu, incl, 31);
      }
      bad = __any_sync(0xffffffffu, bad) || p.offsets[0] != 0;
      if (lane == 0) {
        prefix[p.E] = running;
        *total_tiles = bad ? 0 : running * nb;
        if (bad && blockIdx.x == 0) record_status(p.status, kStatusOffsets, 3);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before either signals the other
  tc_fence_after();
  const uint32_t tmem = warp_bcast(*tmem_base);
  const int total = warp_bcast(*total_tiles);
  const int kchunks = p.K / 64;
  const int kstages = (kchunks + kMmas - 1) / kMmas;

  // The three issuing roles below run with the whole warp: lane 0 waits on
  // the barriers (result broadcast), one elected lane issues.
  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer (both CTAs)
    PipeState<kStages> ps;
    uint32_t issued_mask = 0, last_phase = 0;
    bool ok = true;
    for (int t = pair; t < total && ok; t += npairs) {
      const Tile tl = bcast_tile(tile_of<kEpi>(p, prefix, t));
      const int my_row0 = tl.row0 + (int)rank * BM;
      const int my_brow = leader ? tl.brow0 : tl.brow1;
      for (int ks = 0; ks < kstages; ++ks) {
        if (!mbar_wait_warp(&empty[ps.index], ps.phase ^ 1u, wg, 110)) { ok = false; break; }
        uint8_t* st = stages + ps.index * kStageBytes;
        if (elect_one()) {
          if (leader) mbar_arrive_expect_tx(&full[ps.index], (uint32_t)(2 * G::kStageTx));
          const uint32_t bar = mapa_shared(smem_u32(&full[ps.index]), 0);
          tma_load_2d_pair(st + kOffA, &tmA, bar, ks * kRowBytes, my_row0);
          tma_load_2d_pair(st + kOffB, &tmB, bar, ks * kRowBytes, my_brow);
          // scales: each CTA loads its own rows' block of A scales and both
          // B scale blocks, since each CTA's tensor core reads all 256 of them
          const int x = ks * G::kSfBox;
          tma_load_2d_pair(st + kOffSfa, &tmSfa, bar, x, my_row0 / 128);
          tma_load_2d_pair(st + kOffSfb, &tmSfb, bar, x, tl.brow0 / 128);
          tma_load_2d_pair(st + kOffSfb + kMmas * 512, &tmSfb, bar, x, tl.sfb_blk1);
        }
        __syncwarp();
        issued_mask |= 1u << ps.index;
        last_phase = (last_phase & ~(1u << ps.index)) | (ps.phase << ps.index);
        ps.advance();
      }
    }
    if (leader && lane == 0) {
      // Copies already in flight (both CTAs' loads signal the leader's
      // barriers) land before the pair can exit (after an abort; on the
      // normal path every issued stage has completed already).
      for (int s = 0; s < kStages; ++s)
        if (issued_mask & (1u << s)) mbar_drain(&full[s], (last_phase >> s) & 1u, 100000000ull);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------------ low-rank producer (both CTAs)
    if (kLora) {
      uint32_t phase = 0;
      bool issued = false;
      for (int t = pair; t < total; t += npairs) {
        const Tile tl = bcast_tile(tile_of<kEpi>(p, prefix, t));
        if (!mbar_wait_warp(lora_empty, phase ^ 1u, wg, 120)) break;
        if (elect_one()) {
          if (leader) mbar_arrive_expect_tx(lora_full, (uint32_t)(2 * kLoraBytes));
          const uint32_t bar = mapa_shared(smem_u32(lora_full), 0);
          const int my_row0 = tl.row0 + (int)rank * BM;
          tma_load_2d_pair(lora + kLoraThi, &tmT, bar, 0, my_row0);
          tma_load_2d_pair(lora + kLoraTlo, &tmT, bar, 32, my_row0);
          tma_load_2d_pair(lora + kLoraBl, &tmL, bar, 0, leader ? tl.brow0 : tl.brow1);
        }
        __syncwarp();
        issued = true;
        phase ^= 1u;
      }
      // the last low-rank copies (both CTAs') land before the pair can exit
      if (issued && leader && lane == 0) mbar_drain(lora_full, phase ^ 1u, 100000000ull);
    }
  } else if (warp == 1 && leader) {
    // ------------------------------------------------------------------ MMA issuer (leader only)
    // Descriptors are built once for stage 0 and advanced by byte offset / 16
    // in their start-address field.
    PipeState<kStages> ps;
    uint32_t acc_phase = 0, lora_phase = 0, sf_buf = 0;
    bool ok = true;
    const uint64_t dA = smem_desc(smem_u32(stages + kOffA), 16, kSbo, G::kLayout);
    const uint64_t dB = smem_desc(smem_u32(stages + kOffB), 16, kSbo, G::kLayout);
    const uint64_t dSfa = smem_desc(smem_u32(stages + kOffSfa), 0, 128, kLayoutNone);
    const uint64_t dSfb = smem_desc(smem_u32(stages + kOffSfb), 0, 128, kLayoutNone);
    for (int t = pair; t < total && ok; t += npairs) {
      const bool narrow = (kEpi == kEpiStore && p.E == 0) && warp_bcast(tile_of<kEpi>(p, prefix, t).narrow) != 0;
      const uint32_t idesc_main = narrow ? kIdescMainHalf : kIdescMain;
      if (!mbar_wait_warp(acc_empty, acc_phase ^ 1u, wg, 130)) break;
      tc_fence_after();
      for (int ks = 0; ks < kstages; ++ks) {
        if (!mbar_wait_warp(&full[ps.index], ps.phase, wg, 131)) { ok = false; break; }
        tc_fence_after();
        const int nmma = min(kMmas, kchunks - kMmas * ks);
        const uint64_t so = (uint64_t)((ps.index * kStageBytes) >> 4);
        const uint32_t sf_col = tmem + kTmemSf + sf_buf * kSfColsPerStage;
        if (elect_one()) {
          // each MMA right behind the three scale copies it reads (copies
          // and MMAs run in issue order): with all twelve copies of a stage
          // first, every stage's first MMA waited for all of them
          // (8192^3: 0.1826 -> 0.1764 ms with the low-rank branch)
#pragma unroll
          for (int j = 0; j < kMmas; ++j) {
            if (j < nmma) {
              const uint32_t col = sf_col + j * kSfColsPerMma;
              tc_cp_32x128b_warpx4_pair(col, dSfa + so + 32 * j);               // 512 B per block
              tc_cp_32x128b_warpx4_pair(col + 4, dSfb + so + 32 * j);
              tc_cp_32x128b_warpx4_pair(col + 8, dSfb + so + 32 * (kMmas + j));
              mma_mxf4nvf4_pair(tmem + kTmemAcc, dA + so + 2 * j, dB + so + 2 * j, idesc_main, col, col + 4,
                                (ks > 0 || j > 0) ? 1u : 0u);                    // 32 B of K per MMA
            }
          }
          tc_commit_pair_multicast(&empty[ps.index], 0x3);
        }
        __syncwarp();
        sf_buf ^= 1u;
        ps.advance();
      }
      if (!ok) break;
      if (kLora) {
        if (!mbar_wait_warp(lora_full, lora_phase, wg, 132)) break;
        tc_fence_after();
        if (elect_one()) {
          const uint32_t thi = smem_u32(lora + kLoraThi), tlo = smem_u32(lora + kLoraTlo);
          const uint32_t bl = smem_u32(lora + kLoraBl);
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            const uint32_t ta = part == 0 ? thi : tlo;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
              mma_bf16_pair(tmem + kTmemAcc, smem_desc(ta + 32 * kk, 16, 512, kLayoutSw64),
                            smem_desc(bl + 32 * kk, 16, 512, kLayoutSw64), narrow ? kIdescLoraHalf : kIdescLora, 1u);
          }
          tc_commit_pair_multicast(lora_empty, 0x3);
        }
        __syncwarp();
        lora_phase ^= 1u;
      }
      if (elect_one()) tc_commit_pair_multicast(acc_full, 0x3);
      __syncwarp();
      acc_phase ^= 1u;
    }
    if (elect_one()) {
      tc_commit_pair_local(drain);
      mbar_drain(drain, 0, 1000000000ull);
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------------ epilogue (both CTAs, own rows)
    const int q = warp % 4;
    const int half = (warp - kEpiWarp0) / 4;
    const int r_in_tile = (int)rank * BM + q * 32 + lane;  // row within the pair tile
    const uint32_t acc_empty_leader = mapa_shared(smem_u32(acc_empty), 0);
    uint32_t acc_phase = 0;
    // One 32 x 32-byte box: each lane writes its row (two 16-byte halves in
    // the swizzled order), then one lane hands the box to TMA.  The buffer is
    // reused once TMA has read the previous box.
    constexpr int kRowW = Box::kRowW;
    const uint32_t sbuf = smem_u32(estage + (warp - kEpiWarp0) * Box::kBytes);
    const uint32_t swz = kLora ? (uint32_t)((lane >> 2) & 1) : (uint32_t)((lane >> 1) & 3);
    auto stage_and_store = [&](const uint32_t (&w)[kRowW], int x, int y) {
      if (elect_one()) bulk_wait_read_all();
      __syncwarp();
#pragma unroll
      for (int j = 0; j < kRowW / 4; ++j)
        st_shared_v4(sbuf + lane * Box::kRowBytes + (((uint32_t)j ^ swz) << 4), w[4 * j], w[4 * j + 1], w[4 * j + 2],
                     w[4 * j + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (elect_one()) {
        tma_store_2d(&tmO, estage + (warp - kEpiWarp0) * Box::kBytes, x, y);
        bulk_commit_group();
      }
      __syncwarp();
    };
    for (int t = pair; t < total; t += npairs) {
      const Tile tl = tile_of<kEpi>(p, prefix, t);
      int ok = 1;
      if (lane == 0) ok = mbar_wait(acc_full, acc_phase, wg, 140) ? 1 : 0;
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
      if (lane == 0) mbar_arrive_cluster(acc_empty_leader);
      acc_phase ^= 1u;

      const bool row_ok = r_in_tile < tl.rows;
      const int64_t row = (int64_t)tl.row0 + r_in_tile;
      if (kEpi == kEpiSwiglu) {
        // h = bf16(silu(g) * u); padding rows of the segment inside the pair
        // tile are written as zeros.  Boxes of 32 rows past the segment's
        // 128-aligned extent belong to the next expert and are skipped.
        const int col = tl.col0 + 64 * half;
        const int box_r = (int)rank * BM + q * 32;  // first row of this warp's box, in the tile
        const int row_box = tl.row0 + box_r;
        if (box_r < ((tl.rows + 127) / 128) * 128 && row_box < p.M) {
#pragma unroll
          for (int cc = 0; cc < 64 / (2 * kRowW); ++cc) {  // 2 kRowW columns per box
            uint32_t w[kRowW];
#pragma unroll
            for (int i = 0; i < kRowW; ++i) {
              float hv[2];
#pragma unroll
              for (int k2 = 0; k2 < 2; ++k2) {
                const int c = cc * 2 * kRowW + 2 * i + k2;
                const float g = __uint_as_float(v[c / 32][c % 32]);
                const float u = __uint_as_float(v[2 + c / 32][c % 32]);
                hv[k2] = row_ok ? (g / (1.0f + __expf(-g))) * u : 0.0f;
              }
              w[i] = pack_bf16x2(hv[0], hv[1]);
            }
            stage_and_store(w, col + cc * 2 * kRowW, row_box);
          }
        }
      } else if (kEpi == kEpiSwigluQ4) {
        // h = bf16(silu(g) * u) quantized in place, as q4_quantize would do
        // it: this warp's 64 columns are one 64-element chunk of h, four
        // groups of 16 per lane (its row).  Codes: 32 bytes per row; scales:
        // one 32-bit word (group g in byte g) at the row's place in the MMA
        // scale layout.  Rows follow the SWIGLU rule (padding rows of the
        // segment get zero codes and scales; rows past its 128-aligned end
        // belong to the next expert).
        const int col = tl.col0 + 64 * half;
        if (r_in_tile < ((tl.rows + 127) / 128) * 128 && row < p.M) {
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
        }
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
        // out[r, n] = weight_of[r] * y[r, n] (fp32) in 32-row boxes; boxes
        // holding only rows past the expert's count are not written (padding
        // rows inside a written box carry weight 0 and become zeros)
        const int col = tl.col0 + 128 * half;
        const int box_r = (int)rank * BM + q * 32;
        const int row_box = tl.row0 + box_r;
        if (box_r < tl.rows && row_box < p.M && col < p.N) {
          const float wt = row < p.M ? p.weight_of[row] : 0.0f;
#pragma unroll
          for (int cc = 0; cc < 128 / kRowW; ++cc) {  // kRowW columns per box
            uint32_t w[kRowW];
#pragma unroll
            for (int i = 0; i < kRowW; ++i)
              w[i] = __float_as_uint(wt * __uint_as_float(v[(cc * kRowW + i) / 32][(cc * kRowW + i) % 32]));
            stage_and_store(w, col + cc * kRowW, row_box);
          }
        }
      } else if (kEpi == kEpiStore) {
        const int col = tl.col0 + 128 * half;
        auto value = [&](int c) {  // output column col + c of this lane's row
          float a = __uint_as_float(v[c / 32][c % 32]);
          float sc = alpha_ts;
          if (p.col_scale) sc *= p.col_scale[col + c];
          a *= sc;
          if (p.bias) a += __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.bias)[col + c]);
          return a;
        };
        if (p.E == 0) {
          // dense: boxes of 32 rows x 32 bytes through the warp's staging buffer
          // (a half tile has only accumulator columns [0, 128))
          const int row_box = tl.row0 + (int)rank * BM + q * 32;
          if (row_box < p.M && col < p.N && !(tl.narrow && half)) {
            if (p.out_bf16) {
#pragma unroll
              for (int cc = 0; cc < 128 / (2 * kRowW); ++cc) {  // 2 kRowW columns per box
                uint32_t w[kRowW];
#pragma unroll
                for (int i = 0; i < kRowW; ++i)
                  w[i] = pack_bf16x2(value(cc * 2 * kRowW + 2 * i), value(cc * 2 * kRowW + 2 * i + 1));
                stage_and_store(w, col + cc * 2 * kRowW, row_box);
              }
            } else {
#pragma unroll
              for (int cc = 0; cc < 128 / kRowW; ++cc) {  // kRowW columns per box
                uint32_t w[kRowW];
#pragma unroll
                for (int i = 0; i < kRowW; ++i) w[i] = __float_as_uint(value(cc * kRowW + i));
                stage_and_store(w, col + cc * kRowW, row_box);
              }
            }
          }
        } else if (row_ok && row < p.M && col < p.N) {
          // grouped: rows past the expert's count are not written
#pragma unroll
          for (int c = 0; c < 128; c += 8) {
            float y[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) y[i] = value(c + i);
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
    // the output boxes handed to TMA are written before the CTA exits
    if (elect_one()) bulk_wait_all();
    __syncwarp();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA frees tensor memory or exits while the pair may still touch it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemAlloc);
  }
}

template <int BK, bool kLora, int kEpi>
static cudaError_t launch_one(const Fp4PairLaunch& L, cudaStream_t stream) {
  using G = PGeo<BK>;
  constexpr int kStages = kLora ? G::kStagesLora : G::kStagesNoLora;
  auto kern = fp4_pair_kernel<BK, kStages, kLora, kEpi>;
  const int smem = fp4_smem_total(kLora ? G::kShapeLora : G::kShapeNoLora, kStages) + kAlign;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, (unsigned)L.grid, kThreads, (size_t)smem, stream, 2, L.base.tmA, L.base.tmB, L.base.tmT,
                       L.base.tmL, L.tmSfa, L.tmSfb, L.tmO, L.base.p);
}

template <int BK>
static cudaError_t launch_bk(const Fp4PairLaunch& L, cudaStream_t stream) {
  if (L.base.lora) {
    if (L.base.epilogue != kEpiStore) return cudaErrorInvalidValue;
    return launch_one<BK, true, kEpiStore>(L, stream);
  }
  switch (L.base.epilogue) {
    case kEpiStore: return launch_one<BK, false, kEpiStore>(L, stream);
    case kEpiSwiglu: return launch_one<BK, false, kEpiSwiglu>(L, stream);
    case kEpiSwigluQ4: return launch_one<BK, false, kEpiSwigluQ4>(L, stream);
    case kEpiCombine: return launch_one<BK, false, kEpiCombine>(L, stream);
    case kEpiRows: return launch_one<BK, false, kEpiRows>(L, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fp4pair

cudaError_t launch_fp4_pair_gemm(const Fp4PairLaunch& L, cudaStream_t stream) {
  if (L.grid <= 0 || (L.grid & 1)) return cudaErrorInvalidValue;
  if (L.base.bk == 256) return fp4pair::launch_bk<256>(L, stream);
  if (L.base.bk == 128) return fp4pair::launch_bk<128>(L, stream);
  return cudaErrorInvalidValue;
}

int fp4_pair_stages(bool lora, int bk) {
  if (bk == 256) return lora ? fp4pair::PGeo<256>::kStagesLora : fp4pair::PGeo<256>::kStagesNoLora;
  return lora ? fp4pair::PGeo<128>::kStagesLora : fp4pair::PGeo<128>::kStagesNoLora;
}

}  // namespace bsk
