// gemm_fp8_grouped.cu -- FP8 e4m3 GEMM grouped over MoE experts for sm_103a.
//
//   Y[r, n] = sum_kb sa[kb, r] * sb[(e Nw + n) / 128, kb] * sum_{k in kb} a[r, k] b[e Nw + n, k]
//
// for every row r of expert e's segment ("DeepGEMM teardown (FP8 GEMM)",
// section 5.3: the grouped contiguous layout, each expert's tokens contiguous
// and aligned to whole 128-row blocks, located by group offsets; section 2.2:
// 1x128 activation and 128x128 weight scales; "DeepGEMM for Hopper MoE",
// section 2.1: C = TC(A_fp8, B_fp8) * (sA * sB) per expert).
//
// Orientation: the tokens of one 128-row block of an expert segment are the
// MMA's M (tensor-memory lanes), BN = 128 rows of the expert's weights its N.
// Each thread of the epilogue then owns one token row, so the token scale of
// a K block is one value per thread and the weight scale one per column half:
// promotion costs one multiply per K block plus one FMA per element.
//
// The fp32 scales are applied per 128-wide K block as in the dense FP8 kernel:
// the tensor core writes each K block's partial product into one of four
// tensor-memory slots, the epilogue warps fold it into registers with
// sa[kb, r] * sb[., kb] and hand the slot back.
//
// Tiles: expert by expert, column block by column block, row block by row
// block; a persistent CTA takes tiles c, c + G, ...  The tile table (row
// blocks per expert, prefix-summed) is built on the device from the offsets
// the dispatch kernel wrote, after the dependency wait.
//
// Epilogues:
//   STORE   out[r, n] = y                      (rows of the segment only)
//   ROWS    out fp32 [r, n] = weight_of[r] * y (rows of the segment only)
//   SWIGLU  the tile's weight rows are 64 gate rows f0 .. f0+63 of the expert
//           followed by the 64 up rows F + f0 ..; out bf16 [r, f] =
//           bf16(silu(g) * u) for every row of the segment's 128-row blocks
//           (padding rows as 0).
//
// Roles (384 threads):
//   warp 0      TMA producer: token tile [128 x 128] + two weight boxes [64 x 128]
//   warp 1      tensor-memory allocator, MMA issuer (kind::f8f6f4, K = 32 each)
//   warp 2      tile table
//   warps 4-11  promotion / epilogue: two warps per 32-lane quarter; each
//               thread holds two groups of 32 columns of its token row
#include "budget.hpp"
#include "kernels.h"
#include "ptx.cuh"

namespace bsk {
namespace fp8g {

constexpr int BM = 128;   // token rows per tile (MMA M)
constexpr int BK = 128;   // K per stage = one scale block
constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;
constexpr int kMaxExperts = 1024;
constexpr int kMisc = 2048 + (kMaxExperts + 1) * 4 + 2048;  // barriers, tile table, slack
constexpr int kMaxStages = 12;
constexpr int KBC = 16;   // K blocks whose scales are staged together

template <int BN>
struct Cfg {
  static constexpr int kStageBytes = round_up(BM * BK + BN * BK, kAlign);
  // two staging buffers of [KBC][BM] token scales + [2][KBC] weight scales
  static constexpr int kScaleBytes = round_up(2 * (KBC * BM + 2 * KBC) * 4, kAlign);
  static constexpr int kFit = (kSmemPerCta - kScaleBytes - kMisc - kAlign) / kStageBytes;
  static constexpr int kStages = kFit < kMaxStages ? kFit : kMaxStages;
  static constexpr int kSmem = kStages * kStageBytes + kScaleBytes + kMisc + kAlign;
  static constexpr int kSlots = 512 / BN;   // per-K-block partial slots
  static constexpr int kTmemCols = 512;
  static constexpr int NG = BN / 4;         // columns per thread group (two groups per thread)
  static_assert(kStages >= 3, "ring too shallow");
  static_assert(kSmem <= kSmemPerCta, "smem budget");
  static_assert(kSlots >= 2 && kSlots * BN <= kTmemCols, "tmem budget");
};

struct Tile {
  int row0, rows;     // first token row of the block, rows of the segment in it
  int col0;           // first output column (SWIGLU: first h column)
  int brow0, brow1;   // first weight row of each half of the B tile
  int sb0, sb1;       // weight-scale block row of each half
};

template <int BN, int kEpi>
__device__ __forceinline__ int n_blocks(const Fp8GroupedParams& p) {
  return kEpi == kEpiSwiglu ? p.N / (BN / 2) : (p.N + BN - 1) / BN;
}

// prefix[e] = 128-row blocks of experts 0 .. e-1 (prefix[E] = all of them).
template <int BN, int kEpi>
__device__ __forceinline__ Tile tile_of(const Fp8GroupedParams& p, const int* prefix, int t) {
  const int nbk = n_blocks<BN, kEpi>(p);
  int lo = 0, hi = p.E - 1;  // largest e with prefix[e] * nbk <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] * nbk <= t) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int mblk = prefix[e + 1] - prefix[e];
  const int local = t - prefix[e] * nbk;
  const int nb = local / mblk, mb = local % mblk;
  Tile tl;
  tl.row0 = p.offsets[e] + mb * BM;
  tl.rows = min(BM, p.counts[e] - mb * BM);
  const int wrows = kEpi == kEpiSwiglu ? 2 * p.N : p.N;   // weight rows per expert
  if (kEpi == kEpiSwiglu) {
    tl.col0 = nb * (BN / 2);
    tl.brow0 = e * wrows + nb * (BN / 2);          // gate rows
    tl.brow1 = e * wrows + p.N + nb * (BN / 2);    // up rows
    tl.sb1 = tl.brow1 / 128;
  } else {
    tl.col0 = nb * BN;
    tl.brow0 = e * wrows + nb * BN;
    tl.brow1 = tl.brow0 + BN / 2;
    // a second half past the expert's last column is never stored: keep its
    // scale row inside the expert
    tl.sb1 = (nb * BN + BN / 2 < p.N) ? tl.brow1 / 128 : tl.brow0 / 128;
  }
  tl.sb0 = tl.brow0 / 128;
  return tl;
}

template <int BN, int kEpi>
__global__ void __launch_bounds__(kThreads, 1)
    fp8_grouped_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const Fp8GroupedParams p) {
  using C = Cfg<BN>;
  constexpr int NG = C::NG;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + kAlign - 1) &
                                             ~static_cast<uintptr_t>(kAlign - 1));
  uint8_t* stages = base;
  float* ssa = reinterpret_cast<float*>(base + C::kStages * C::kStageBytes);  // [2][KBC][BM]
  float* ssb = ssa + 2 * KBC * BM;                                            // [2][2][KBC]
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::kStages * C::kStageBytes + C::kScaleBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::kStages;
  uint64_t* pfull = bars + 2 * C::kStages;   // [kSlots] partial written by the tensor core
  uint64_t* pempty = pfull + C::kSlots;      // [kSlots] partial read by the epilogue
  uint64_t* drain = pfull + 2 * C::kSlots;
  uint32_t* tmem_base = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_i = reinterpret_cast<int*>(tmem_base + 1);
  int* total_s = abort_i + 1;
  int* prefix = total_s + 1;                 // [E + 1]
  volatile int* abort_flag = abort_i;
  const WaitGuard wg{abort_flag, p.status, p.wait_ns};
  const int warp = warp_bcast((int)(threadIdx.x / 32)), lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    griddep_launch_dependents();
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < C::kSlots; ++i) {
      mbar_init(&pfull[i], 1);
      mbar_init(&pempty[i], 8);  // one arrive per epilogue warp
    }
    mbar_init(drain, 1);
    *abort_i = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  // Everything above touched only this CTA's own resources; the operands and
  // the offset table come from the kernels before this one on the stream.
  griddep_wait();
  if (warp == 2) {
    // Tile table: validate the offsets and prefix-sum the row blocks.
    int running = 0;
    bool bad = false;
    for (int e0 = 0; e0 < p.E; e0 += 32) {
      const int e = e0 + lane;
      int blocks = 0;
      if (e < p.E) {
        const int off = p.offsets[e], cnt = p.counts[e], nxt = p.offsets[e + 1];
        if (cnt < 0 || (off % BM) != 0 || off + cnt > nxt || nxt > p.M) bad = true;
        blocks = (max(cnt, 0) + BM - 1) / BM;
      }
      int incl = blocks;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
      }
      if (e < p.E) prefix[e] = running + incl - blocks;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    bad = __any_sync(0xffffffffu, bad) || p.offsets[0] != 0;
    if (lane == 0) {
      prefix[p.E] = running;
      *total_s = bad ? 0 : running * n_blocks<BN, kEpi>(p);
      if (bad && blockIdx.x == 0) record_status(p.status, kStatusOffsets, 2);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = warp_bcast(*tmem_base);
  const int total = warp_bcast(*total_s);
  const int nkb = p.K / BK;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    PipeState<C::kStages> ps;
    uint32_t issued_mask = 0, last_phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile tl = tile_of<BN, kEpi>(p, prefix, t);
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait_warp(&empty[ps.index], ps.phase ^ 1u, wg, 300)) { ok = false; break; }
        uint8_t* st = stages + ps.index * C::kStageBytes;
        if (elect_one()) {
          mbar_arrive_expect_tx(&full[ps.index], (uint32_t)(BM * BK + BN * BK));
          tma_load_2d(st, &tmA, &full[ps.index], kb * BK, tl.row0);
          tma_load_2d(st + BM * BK, &tmB, &full[ps.index], kb * BK, tl.brow0);
          tma_load_2d(st + BM * BK + (BN / 2) * BK, &tmB, &full[ps.index], kb * BK, tl.brow1);
        }
        __syncwarp();
        issued_mask |= 1u << ps.index;
        last_phase = (last_phase & ~(1u << ps.index)) | (ps.phase << ps.index);
        ps.advance();
      }
    }
    if (lane == 0) {
      // copies already in flight land before the CTA can exit
      for (int s = 0; s < C::kStages; ++s)
        if (issued_mask & (1u << s)) mbar_drain(&full[s], (last_phase >> s) & 1u, 100000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    PipeState<C::kStages> ps;
    PipeState<C::kSlots> sl;
    constexpr uint32_t idesc = idesc_e4m3(BM, BN);
    const uint64_t dA = smem_desc(smem_u32(stages), 16, 1024, kLayoutSw128);
    const uint64_t dB = smem_desc(smem_u32(stages + BM * BK), 16, 1024, kLayoutSw128);
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait_warp(&pempty[sl.index], sl.phase ^ 1u, wg, 310)) { ok = false; break; }
        if (!mbar_wait_warp(&full[ps.index], ps.phase, wg, 311)) { ok = false; break; }
        tc_fence_after();
        const uint64_t so = (uint64_t)((ps.index * C::kStageBytes) >> 4);
        const uint32_t d = tmem + sl.index * BN;
        if (elect_one()) {
#pragma unroll
          for (int j = 0; j < BK / 32; ++j)
            mma_e4m3(d, dA + so + 2 * j, dB + so + 2 * j, idesc, j > 0 ? 1u : 0u);  // 32 B of K per MMA
          tc_commit(&empty[ps.index]);
          tc_commit(&pfull[sl.index]);
        }
        __syncwarp();
        ps.advance();
        sl.advance();
      }
    }
    if (elect_one()) {
      tc_commit(drain);
      mbar_drain(drain, 0, 1000000000ull);
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------------ promotion + epilogue
    // Walks (tile, chunk of KBC K blocks) in order; the next chunk's scales
    // are staged with cp.async while this one is promoted.  After an abort the
    // warps keep walking (skipping waits and work) so the named barriers of
    // all eight warps still match.
    const int q = warp % 4, half = (warp - kEpiWarp0) / 4;
    const int r = q * 32 + lane;                     // token row within the tile
    const int etid = threadIdx.x - kEpiWarp0 * 32;  // 0 .. 255
    // this thread's two column groups and the weight-scale half of each
    const int c0 = kEpi == kEpiSwiglu ? half * NG : half * (BN / 2);
    const int c1 = kEpi == kEpiSwiglu ? BN / 2 + half * NG : half * (BN / 2) + NG;
    const int g0 = kEpi == kEpiSwiglu ? 0 : half;
    const int g1 = kEpi == kEpiSwiglu ? 1 : half;
    const int nchunks = (nkb + KBC - 1) / KBC;
    PipeState<C::kSlots> sl;
    bool ok = true;
    auto stage_scales = [&](const Tile& tl, int c, int buf) {
      float* da = ssa + buf * KBC * BM;
      float* db = ssb + buf * 2 * KBC;
      for (int i = etid; i < KBC * BM; i += 256) {
        const int kbl = i / BM, m = i % BM;
        const int kb = c * KBC + kbl, row = tl.row0 + m;
        const bool valid = kb < nkb && row < p.M;
        const float* src = valid ? p.sfa + (size_t)kb * p.M + row : p.sfa;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(da + i)), "l"(src),
                     "r"(valid ? 4 : 0)
                     : "memory");
      }
      for (int i = etid; i < 2 * KBC; i += 256) {
        const int hh = i / KBC, kb = c * KBC + i % KBC;
        const bool valid = kb < nkb;
        const float* src = valid ? p.sfb + (size_t)(hh ? tl.sb1 : tl.sb0) * nkb + kb : p.sfb;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(db + i)), "l"(src),
                     "r"(valid ? 4 : 0)
                     : "memory");
      }
    };
    auto store_tile = [&](const Tile& tl, const float (&a0)[NG], const float (&a1)[NG]) {
      const long long row = (long long)tl.row0 + r;
      const bool row_ok = r < tl.rows;
      if (row >= p.M) return;
      if constexpr (kEpi == kEpiSwiglu) {
        // h = bf16(silu(g) * u); padding rows of the segment are written as 0
        uint16_t* out = reinterpret_cast<uint16_t*>(p.out) + row * p.ldo + tl.col0 + half * NG;
#pragma unroll
        for (int c = 0; c < NG; c += 8) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float hv[2];
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
              const float g = a0[c + 2 * i + k2], u = a1[c + 2 * i + k2];
              hv[k2] = row_ok ? (g / (1.0f + __expf(-g))) * u : 0.0f;
            }
            w[i] = pack_bf16x2(hv[0], hv[1]);
          }
          *reinterpret_cast<uint4*>(out + c) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      } else {
        if (!row_ok) return;
        const float wt = kEpi == kEpiRows ? __ldg(p.weight_of + row) : 1.0f;
#pragma unroll
        for (int gi = 0; gi < 2; ++gi) {
          const int col = tl.col0 + (gi ? c1 : c0);
          if (col >= p.N) continue;
          const float* a = gi ? a1 : a0;
          if (p.out_bf16) {
            uint16_t* out = reinterpret_cast<uint16_t*>(p.out) + row * p.ldo + col;
#pragma unroll
            for (int c = 0; c < NG; c += 8) {
              uint32_t w[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) w[i] = pack_bf16x2(wt * a[c + 2 * i], wt * a[c + 2 * i + 1]);
              *reinterpret_cast<uint4*>(out + c) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
            float4* out = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + row * p.ldo + col);
#pragma unroll
            for (int c = 0; c < NG; c += 4)
              out[c / 4] = make_float4(wt * a[c], wt * a[c + 1], wt * a[c + 2], wt * a[c + 3]);
          }
        }
      }
    };

    int t = blockIdx.x;
    bool have = t < total;
    Tile tl = {};
    if (have) {
      tl = tile_of<BN, kEpi>(p, prefix, t);
      stage_scales(tl, 0, 0);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    float acc0[NG], acc1[NG];
#pragma unroll
    for (int i = 0; i < NG; ++i) acc0[i] = acc1[i] = 0.0f;
    int c = 0, qi = 0;
    while (have) {
      Tile tn = tl;
      int tnext = t, cn = c + 1;
      bool haven = true;
      if (cn == nchunks) {
        cn = 0;
        tnext = t + gridDim.x;
        haven = tnext < total;
        if (haven) tn = tile_of<BN, kEpi>(p, prefix, tnext);
      }
      if (haven) stage_scales(tn, cn, (qi + 1) & 1);
      asm volatile("cp.async.commit_group;" ::: "memory");
      asm volatile("cp.async.wait_group 1;" ::: "memory");
      asm volatile("bar.sync 1, 256;" ::: "memory");
      const float* csa = ssa + (qi & 1) * KBC * BM;
      const float* csb = ssb + (qi & 1) * 2 * KBC;
      const int kc0 = c * KBC;
      const int kb_end = min(nkb, kc0 + KBC);
      for (int kb = kc0; kb < kb_end; ++kb) {
        if (ok) {
          int w_ok = 1;
          if (lane == 0) w_ok = mbar_wait(&pfull[sl.index], sl.phase, wg, 320) ? 1 : 0;
          ok = __shfl_sync(0xffffffffu, w_ok, 0) != 0;
        }
        if (ok) {
          tc_fence_after();
          const float sa = csa[(kb - kc0) * BM + r];
          const float s0 = sa * csb[g0 * KBC + kb - kc0];
          const float s1 = sa * csb[g1 * KBC + kb - kc0];
          const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16) + sl.index * BN;
          uint32_t v0[NG], v1[NG];
          tmem_ld_cols<NG>(lane_base + c0, v0);
          tmem_ld_cols<NG>(lane_base + c1, v1);
          tmem_ld_wait();
          // every column of the slot this warp reads is in registers: hand it back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&pempty[sl.index]);
#pragma unroll
          for (int i = 0; i < NG; ++i) {
            acc0[i] = fmaf(__uint_as_float(v0[i]), s0, acc0[i]);
            acc1[i] = fmaf(__uint_as_float(v1[i]), s1, acc1[i]);
          }
        }
        sl.advance();
      }
      if (cn == 0) {
        // the tile's last chunk: store, reset the accumulators
        if (ok) store_tile(tl, acc0, acc1);
#pragma unroll
        for (int i = 0; i < NG; ++i) acc0[i] = acc1[i] = 0.0f;
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");  // this scale buffer may be refilled next
      tl = tn;
      t = tnext;
      c = cn;
      have = haven;
      ++qi;
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int BN, int kEpi>
static cudaError_t launch_epi(const Fp8GroupedLaunch& L, cudaStream_t stream) {
  using C = Cfg<BN>;
  auto kern = fp8_grouped_kernel<BN, kEpi>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, (unsigned)L.grid, kThreads, (size_t)C::kSmem, stream, 1, L.tmA, L.tmB, L.p);
}

}  // namespace fp8g

int fp8_grouped_stages() { return fp8g::Cfg<kFp8GroupedBN>::kStages; }

cudaError_t launch_fp8_grouped(const Fp8GroupedLaunch& L, cudaStream_t stream) {
  if (L.grid <= 0 || L.p.E <= 0 || L.p.E > fp8g::kMaxExperts) return cudaErrorInvalidValue;
  switch (L.epilogue) {
    case kEpiStore: return fp8g::launch_epi<kFp8GroupedBN, kEpiStore>(L, stream);
    case kEpiSwiglu: return fp8g::launch_epi<kFp8GroupedBN, kEpiSwiglu>(L, stream);
    case kEpiRows: return fp8g::launch_epi<kFp8GroupedBN, kEpiRows>(L, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace bsk
