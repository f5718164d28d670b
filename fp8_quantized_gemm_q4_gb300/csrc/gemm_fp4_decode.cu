// gemm_fp4_decode.cu -- block-scaled FP4 GEMM for decode shapes (M <= 32) on sm_103a.
//
//   Y[m,n] = alpha * ts * col_scale[n] * sum_g sx[m,g] sw[n,g] sum_{k in g} x w + bias[n]
//   ("Warp-specialised W4A4 kernel on the newest GPU architecture", section 1)
//
// A decode step reads every weight once and does little arithmetic with it
// ("Tencent AI Infra interview notes", decode intensity: 2KN FLOPs against
// KN * bytes_per_weight, 4 FLOP/byte for 4-bit weights), so what counts is
// streaming the weights through every SM.  Swap-AB: the weight rows fill the
// MMA's M = 128, the M <= 32 tokens are its N (16 or 32), so the tensor core
// runs full-height block-scaled MMAs (kind::mxf4nvf4, block16 ue4m3 scales
// applied by the tensor core: no promotion) over the weights.
//
// Work units are (weight tile of 128 rows, K stage of 256) pairs; with fewer
// tiles than CTAs they form one sequence shared out evenly over the grid
// (stream-K, "DeepGEMM teardown" sections 1.2 and 3.2: small M leaves SMs
// idle), otherwise the CTAs take whole tiles in turn.  A CTA accumulates its K
// range of a tile in one tensor-memory slot; a tile cut between CTAs is
// finished by the last of them (acquire-release counter in the caller's
// workspace, pieces summed in K order, counter reset), as in the FP8 kernel.
//
// Per stage the producer loads, for one weight tile: W codes [128 x 128 B]
// and X codes [TN x 128 B] through 128B-swizzled tensor maps, and the four
// 512-byte scale tiles of each (the MMA layout keeps a 128-row block's tiles
// of one stage contiguous) with bulk copies.  The MMA warp stages the scales
// in tensor memory with tcgen05.cp (token row n sits at lane n % 32, column
// n / 32 of its tile, so N = TN <= 32 reads column 0) and issues four MMAs.
//
// kMulti: G products Y_g = X W_g^T that share the tokens form one list of
// weight tiles (tile t is tile t mod T of product t / T, T = tiles of one
// product) under one stream-K schedule, each product with its own weight map,
// scales and output, so a decode step's projections pay the launch, first
// loads and fix-up tail once.
#include "budget.hpp"
#include "kernels.h"
#include "ptx.cuh"

namespace bsk {
namespace fp4dec {

constexpr int BM = 128;          // weight rows per tile (MMA M)
constexpr int BK = 256;          // FP4 elements of K per stage
constexpr int kRowBytes = BK / 2;
constexpr int kMmas = BK / 64;   // K = 64 per MMA
constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;
constexpr int kMisc = 2048;
constexpr int kMaxStages = 12;
constexpr int kSfColsPerMma = 8;           // 4 columns of weight scales, 4 of token scales
constexpr int kSfCols = 2 * kMmas * kSfColsPerMma;  // two stage buffers

template <int TN>
struct Cfg {
  static constexpr int kOffW = 0;
  static constexpr int kOffX = BM * kRowBytes;
  static constexpr int kOffSfw = kOffX + TN * kRowBytes;
  static constexpr int kOffSfx = kOffSfw + kMmas * 512;
  static constexpr int kStageBytes = round_up(kOffSfx + kMmas * 512, kAlign);
  static constexpr int kTx = kOffSfx + kMmas * 512;   // bytes one stage's copies deliver
  // TN 16: a 5-stage ring (about 113 KB) and at most 85 registers a thread,
  // so that two CTAs share an SM and a GEMM launched behind this one streams
  // its first weight stages while this one finishes
  static constexpr int kMax = TN == 16 ? 5 : kMaxStages;
  static constexpr int kStages =
      (kSmemPerCta - kMisc - kAlign) / kStageBytes < kMax ? (kSmemPerCta - kMisc - kAlign) / kStageBytes : kMax;
  static constexpr int kSmem = kStages * kStageBytes + kMisc + kAlign;
  static constexpr int kSlots = 8;                     // accumulator slots (one per segment)
  static constexpr int kTmemAcc = 0;
  static constexpr int kTmemSf = kSlots * TN;
  static constexpr int kTmemCols = pow2_cols(kSlots * TN + kSfCols);
  static constexpr int kColsPerWarp = TN / 2;
  static_assert(kStages >= 2, "ring too shallow");
  static_assert(kSmem <= kSmemPerCta, "smem budget");
  static_assert(kTmemCols <= bsk::kTmemCols, "tmem budget");
  static_assert(kOffX % 1024 == 0 && kOffSfw % 16 == 0, "stage alignment");
};

struct Seg {
  int t, kb0, kb1;  // weight tile t, K stages [kb0, kb1)
};

// A CTA's share of the (tile, K stage) sequence.  With at least as many tiles
// as CTAs, whole tiles t = c, c + G, ... (no tile is cut, no fix-up runs; two
// CTAs of an SM, c and c + G / 2, then hold at most one tile more than the
// average between them); with fewer, one contiguous stream-K range.
struct Walk {
  long long cur, end;
  int step;  // > 0: whole tiles, cur / end count tiles; 0: stream-K, they count units
  __device__ __forceinline__ Walk(int total, int nks) {
    if (total >= (int)gridDim.x) {
      cur = blockIdx.x;
      end = total;
      step = (int)gridDim.x;
    } else {
      const long long U = (long long)total * nks;
      cur = (long long)blockIdx.x * U / gridDim.x;
      end = (long long)(blockIdx.x + 1) * U / gridDim.x;
      step = 0;
    }
  }
  __device__ __forceinline__ bool next(int nks, Seg& s) {
    if (cur >= end) return false;
    if (step) {
      s.t = (int)cur;
      s.kb0 = 0;
      s.kb1 = nks;
      cur += step;
      return true;
    }
    s.t = (int)(cur / nks);
    s.kb0 = (int)(cur % nks);
    s.kb1 = (int)min((long long)nks, s.kb0 + (end - cur));
    cur += s.kb1 - s.kb0;
    return true;
  }
};

__device__ __forceinline__ int sk_owner(long long u, long long U, int G) { return (int)(((u + 1) * G - 1) / U); }

template <int TN, bool kMulti>
__global__ void __launch_bounds__(kThreads, TN == 16 ? 2 : 1)
    fp4_decode_kernel(const __grid_constant__ typename WArg<kMulti>::type tmW,
                      const __grid_constant__ CUtensorMap tmX, const Fp4DecodeParams p) {
  using C = Cfg<TN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + kAlign - 1) &
                                             ~static_cast<uintptr_t>(kAlign - 1));
  uint8_t* stages = base;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::kStages * C::kStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::kStages;
  uint64_t* pfull = bars + 2 * C::kStages;
  uint64_t* pempty = pfull + C::kSlots;
  uint64_t* drain = pfull + 2 * C::kSlots;
  uint32_t* tmem_base = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_i = reinterpret_cast<int*>(tmem_base + 1);
  int* fix_flag = abort_i + 1;
  volatile int* abort_flag = abort_i;
  const WaitGuard wg{abort_flag, p.status, p.wait_ns};
  const int warp = warp_bcast((int)(threadIdx.x / 32)), lane = threadIdx.x % 32;

  // Prologue: the producer initialises the barriers and starts loading; the
  // tensor-memory allocation overlaps its first loads (named barrier 2).
  uint32_t tmem = 0;
  if (warp == 0) {
    if (lane == 0) {
      griddep_launch_dependents();
      for (int s = 0; s < C::kStages; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], 1);
      }
      for (int i = 0; i < C::kSlots; ++i) {
        mbar_init(&pfull[i], 1);
        mbar_init(&pempty[i], 8);
      }
      mbar_init(drain, 1);
      *abort_i = 0;
      fence_barrier_init();
      if constexpr (kMulti) {
        for (int g = 0; g < p.G; ++g) prefetch_tmap(&tmW.m[g]);
      } else {
        prefetch_tmap(&tmW);
      }
      prefetch_tmap(&tmX);
    }
    __syncwarp();
    asm volatile("bar.arrive 2, %0;" ::"n"(kThreads) : "memory");
  } else {
    if (warp == 1) {
      tmem_alloc(tmem_base, C::kTmemCols);
      tmem_relinquish();
    }
    tc_fence_before();
    asm volatile("bar.sync 2, %0;" ::"n"(kThreads) : "memory");
    tc_fence_after();
    tmem = warp_bcast(*tmem_base);
  }

  const int per = (p.N + BM - 1) / BM;     // weight tiles of one product (one token block: M <= TN)
  const int total = (kMulti ? p.G : 1) * per;
  const int nks = p.K / BK;                // K stages (K % 256 == 0)
  // tile t: product and weight-row block within it
  auto t_g = [&](int t) { return kMulti ? t / per : 0; };
  auto t_w = [&](int t) { return kMulti ? t % per : t; };
  const int kchunks = p.K / 64;            // 512-byte scale tiles per 128-row block

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    PipeState<C::kStages> ps;
    uint32_t issued_mask = 0, last_phase = 0;
    bool ok = true;
    const int pre = p.pre_b < C::kStages ? p.pre_b : C::kStages;
    int item = 0;
    // token codes and scales of the first `issued` items (ring slots
    // 0 .. issued-1), once the preceding kernel has finished
    auto late_token_loads = [&](int issued) {
      griddep_wait();
      Walk w2(total, nks);
      Seg s2;
      int i = 0;
      while (i < issued && w2.next(nks, s2))
        for (int kb = s2.kb0; kb < s2.kb1 && i < issued; ++kb, ++i)
          if (elect_one()) {
            uint8_t* st = stages + i * C::kStageBytes;
            tma_load_2d(st + C::kOffX, &tmX, &full[i], kb * kRowBytes, 0);
            bulk_load(st + C::kOffSfx, p.sfx + (size_t)kb * kMmas * 512, kMmas * 512, &full[i]);
          }
      __syncwarp();
    };
    if (pre == 0) griddep_wait();
    Walk w(total, nks);
    Seg sg;
    while (ok && w.next(nks, sg)) {
      for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
        if (!mbar_wait_warp(&empty[ps.index], ps.phase ^ 1u, wg, 210)) { ok = false; break; }
        uint8_t* st = stages + ps.index * C::kStageBytes;
        if (elect_one()) {
          mbar_arrive_expect_tx(&full[ps.index], (uint32_t)C::kTx);
          const int g = t_g(sg.t), wt = t_w(sg.t);
          const CUtensorMap* mw;
          if constexpr (kMulti) mw = &tmW.m[g];
          else mw = &tmW;
          const uint8_t* sfw = kMulti ? pick(p.sfw_g, g) : p.sfw;
          tma_load_2d(st + C::kOffW, mw, &full[ps.index], kb * kRowBytes, wt * BM);
          bulk_load(st + C::kOffSfw, sfw + ((size_t)wt * kchunks + (size_t)kb * kMmas) * 512, kMmas * 512,
                    &full[ps.index]);
          if (item >= pre) {
            tma_load_2d(st + C::kOffX, &tmX, &full[ps.index], kb * kRowBytes, 0);
            bulk_load(st + C::kOffSfx, p.sfx + (size_t)kb * kMmas * 512, kMmas * 512, &full[ps.index]);
          }
        }
        __syncwarp();
        issued_mask |= 1u << ps.index;
        last_phase = (last_phase & ~(1u << ps.index)) | (ps.phase << ps.index);
        ps.advance();
        if (++item == pre) late_token_loads(pre);
      }
    }
    if (item < pre) late_token_loads(item);
    if (lane == 0) {
      for (int s = 0; s < C::kStages; ++s)
        if (issued_mask & (1u << s)) mbar_drain(&full[s], (last_phase >> s) & 1u, 100000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    PipeState<C::kStages> ps;
    PipeState<C::kSlots> sl;
    uint32_t sf_buf = 0;
    constexpr uint32_t idesc = idesc_mxf4nvf4(BM, TN);
    const uint64_t dW = smem_desc(smem_u32(stages + C::kOffW), 16, 1024, kLayoutSw128);
    const uint64_t dX = smem_desc(smem_u32(stages + C::kOffX), 16, 1024, kLayoutSw128);
    const uint64_t dSfw = smem_desc(smem_u32(stages + C::kOffSfw), 0, 128, kLayoutNone);
    const uint64_t dSfx = smem_desc(smem_u32(stages + C::kOffSfx), 0, 128, kLayoutNone);
    bool ok = true;
    Walk w(total, nks);
    Seg sg;
    while (ok && w.next(nks, sg)) {
      if (!mbar_wait_warp(&pempty[sl.index], sl.phase ^ 1u, wg, 220)) { ok = false; break; }
      const uint32_t d = tmem + C::kTmemAcc + sl.index * TN;
      for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
        if (!mbar_wait_warp(&full[ps.index], ps.phase, wg, 221)) { ok = false; break; }
        tc_fence_after();
        const uint64_t so = (uint64_t)((ps.index * C::kStageBytes) >> 4);
        const uint32_t sf_col = tmem + C::kTmemSf + sf_buf * kMmas * kSfColsPerMma;
        if (elect_one()) {
#pragma unroll
          for (int j = 0; j < kMmas; ++j) {
            const uint32_t col = sf_col + j * kSfColsPerMma;
            tc_cp_32x128b_warpx4(col, dSfw + so + 32 * j);      // 512 B: weight rows 0..127
            tc_cp_32x128b_warpx4(col + 4, dSfx + so + 32 * j);  // 512 B: token rows 0..127
            mma_mxf4nvf4(d, dW + so + 2 * j, dX + so + 2 * j, idesc, col, col + 4, (kb > sg.kb0 || j > 0) ? 1u : 0u);
          }
          tc_commit(&empty[ps.index]);
        }
        __syncwarp();
        sf_buf ^= 1u;
        ps.advance();
      }
      if (!ok) break;
      if (elect_one()) tc_commit(&pfull[sl.index]);
      __syncwarp();
      sl.advance();
    }
    if (elect_one()) {
      tc_commit(drain);
      mbar_drain(drain, 0, 1000000000ull);
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------------ epilogue
    constexpr int NC = C::kColsPerWarp;
    const int q = warp % 4, half = (warp - kEpiWarp0) / 4;
    const int col0 = half * NC;                      // first token of this warp's columns
    const int r = q * 32 + lane;                     // weight row within the tile
    const int etid = threadIdx.x - kEpiWarp0 * 32;
    griddep_wait();
    const float alpha_ts = p.alpha * (p.a_ts ? __ldg(p.a_ts) : 1.0f) * (p.b_ts ? __ldg(p.b_ts) : 1.0f);
    PipeState<C::kSlots> sl;
    bool ok = true;
    auto store_out = [&](const Seg& s, const float (&y)[NC]) {
      const int n = t_w(s.t) * BM + r;  // weight row = output column
      if (n >= p.N) return;
      void* const out = kMulti ? pick(p.out_g, t_g(s.t)) : p.out;
      const float sc = alpha_ts * (p.col_scale ? __ldg(p.col_scale + n) : 1.0f);
      const float b = p.bias ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.bias)[n]) : 0.0f;
#pragma unroll
      for (int i = 0; i < NC; ++i) {
        const int m = col0 + i;
        if (m < p.M) {
          const float v = y[i] * sc + b;
          if (p.out_bf16)
            reinterpret_cast<__nv_bfloat16*>(out)[(size_t)m * p.ldo + n] = __float2bfloat16_rn(v);
          else
            reinterpret_cast<float*>(out)[(size_t)m * p.ldo + n] = v;
        }
      }
    };
    Walk w(total, nks);
    Seg sg;
    float acc[NC];
    while (w.next(nks, sg)) {
      if (ok) {
        int w_ok = 1;
        if (lane == 0) w_ok = mbar_wait(&pfull[sl.index], sl.phase, wg, 230) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, w_ok, 0) != 0;
      }
      if (ok) {
        tc_fence_after();
        uint32_t v[NC];
        tmem_ld_cols<NC>(tmem + ((uint32_t)(q * 32) << 16) + C::kTmemAcc + sl.index * TN + col0, v);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pempty[sl.index]);
#pragma unroll
        for (int i = 0; i < NC; ++i) acc[i] = __uint_as_float(v[i]);
      } else {
#pragma unroll
        for (int i = 0; i < NC; ++i) acc[i] = 0.0f;
      }
      sl.advance();
      if (sg.kb0 == 0 && sg.kb1 == nks) {
        if (ok) store_out(sg, acc);
        continue;
      }
      // a piece of a tile cut between CTAs (see the file comment)
      const long long U = (long long)total * nks, u0 = (long long)sg.t * nks;
      const int c_first = sk_owner(u0, U, (int)gridDim.x);
      const int n_parts = sk_owner(u0 + nks - 1, U, (int)gridDim.x) - c_first + 1;
      const int j = (int)blockIdx.x - c_first;
      float* parts = p.work + (size_t)sg.t * p.maxc * (BM * TN);
      float4* mine = reinterpret_cast<float4*>(parts + (size_t)j * (BM * TN) + r * TN + col0);
#pragma unroll
      for (int i = 0; i < NC; i += 4) mine[i / 4] = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (etid == 0) {
        int old;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(p.counters + sg.t) : "memory");
        *fix_flag = old == n_parts - 1;
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (*fix_flag) {
#pragma unroll
        for (int i = 0; i < NC; ++i) acc[i] = 0.0f;
        for (int jj = 0; jj < n_parts; ++jj) {
          const float4* src = reinterpret_cast<const float4*>(parts + (size_t)jj * (BM * TN) + r * TN + col0);
#pragma unroll
          for (int i = 0; i < NC; i += 4) {
            const float4 v4 = __ldcg(src + i / 4);
            acc[i] += v4.x;
            acc[i + 1] += v4.y;
            acc[i + 2] += v4.z;
            acc[i + 3] += v4.w;
          }
        }
        if (ok) store_out(sg, acc);
        if (etid == 0) p.counters[sg.t] = 0;
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");  // fix_flag is rewritten by the next piece
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int TN, bool kMulti>
static cudaError_t launch_tn(const Fp4DecodeLaunch& L, cudaStream_t stream) {
  using C = Cfg<TN>;
  auto kern = fp4_decode_kernel<TN, kMulti>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  // all of the SM's unified memory as shared memory, so two decode CTAs fit
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  if constexpr (kMulti)
    return launch_kernel(kern, (unsigned)L.grid, kThreads, (size_t)C::kSmem, stream, 1, L.tmW_g, L.tmX, L.p);
  else
    return launch_kernel(kern, (unsigned)L.grid, kThreads, (size_t)C::kSmem, stream, 1, L.tmW, L.tmX, L.p);
}

}  // namespace fp4dec

int fp4_decode_stages(int tile_n) {
  return tile_n == 16 ? fp4dec::Cfg<16>::kStages : fp4dec::Cfg<32>::kStages;
}

cudaError_t launch_fp4_decode(const Fp4DecodeLaunch& L, cudaStream_t stream) {
  if (L.grid <= 0 || L.p.G < 1 || L.p.G > kMaxProducts) return cudaErrorInvalidValue;
  const bool multi = L.p.G > 1;
  if (L.tile_n == 16) return multi ? fp4dec::launch_tn<16, true>(L, stream) : fp4dec::launch_tn<16, false>(L, stream);
  if (L.tile_n == 32) return multi ? fp4dec::launch_tn<32, true>(L, stream) : fp4dec::launch_tn<32, false>(L, stream);
  return cudaErrorInvalidValue;
}

}  // namespace bsk
