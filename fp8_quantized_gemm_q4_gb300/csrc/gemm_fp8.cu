// gemm_fp8.cu -- FP8 e4m3 GEMM with fp32 block scales for sm_103a.
//
//   Y[m,n] = sum_kb sa[kb,m] * sb[n/128,kb] * sum_{k in kb} a[m,k] b[n,k]
//   ("DeepGEMM for Hopper MoE", section 2.1: C = TC(A_fp8, B_fp8) * (sA * sB);
//    "DeepGEMM teardown (FP8 GEMM)", section 2.2: per-token 1x128 activation
//    and 128x128 weight scales applied inside the kernel; section 2.3: FP32
//    accumulation, conversion only at the output)
//
// The fp32 scales are not a format the tensor core's block scaling takes, so
// they are applied per 128-wide K block ("promotion"): the tensor core writes
// the block's partial product into a ring of tensor-memory slots (up to 16)
// and the epilogue warps fold each into fp32 registers, acc += partial * sb *
// sa, while the tensor core fills the next slots.
//
// Swap-AB orientation for every M: weight rows fill the MMA's M = 128 (one
// weight-scale block per tile), the tokens are the MMA's N (16 .. 128), so the
// decode shapes (M = 1 .. 16, "DeepGEMM teardown" section 1.2: M of 1 to 16
// idles most of a normal tile) stream the weights through full 128-row MMAs.
//
// Work is a list of (tile, K-block range) segments per CTA:
//  - tiles >= CTAs: each persistent CTA takes whole tiles t = c, c + G, ...
//  - tiles <  CTAs (decode: N = 7168 gives 56 weight tiles for 152 SMs):
//    stream-K ("DeepGEMM teardown" sections 1.2 and 3.2: small M leaves SMs
//    idle; wave scheduling).  The tiles' K blocks form one sequence of units
//    u = t * nkb + kb that is cut into G equal contiguous ranges, one per CTA,
//    so every SM streams the same share of the weights.  A tile cut between
//    CTAs is finished by whichever of them arrives last: each writes its fp32
//    partial to the caller's workspace and counts itself in on the tile's
//    counter; the last one sums the partials in the fixed order of their K
//    ranges (deterministic whatever the arrival order), writes the output and
//    resets the counter to zero for the next call.  Nobody waits for anybody.
//
// Roles (384 threads):
//   warp 0      TMA producer: weight tile [128 x 128] + token tile [TN x 128]
//   warp 1      tensor-memory allocator, MMA issuer (tcgen05.mma kind::f8f6f4,
//               K = 32 per instruction)
//   warps 4-11  promotion / epilogue: two warps per 32-lane quarter, each
//               owning half of the TN token columns of its weight rows
//
// Programmatic dependent launch: the prologue runs before griddep_wait().
// With p.pre_b > 0 the producer also issues the weight loads of its first
// p.pre_b stages before waiting (the caller has promised that the kernel
// before this one on the stream does not write the weights or their scales),
// so the weight stream starts while the activation quantizer still runs.
#include "budget.hpp"
#include "kernels.h"
#include "ptx.cuh"

namespace bsk {
namespace fp8 {

constexpr int BM = 128;   // weight rows per tile (MMA M)
constexpr int BK = 128;   // K per stage = one scale block
constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;
constexpr int kMisc = 2048;
constexpr int kMaxStages = 12;

constexpr int KBC = 32;   // K blocks whose scales are staged together
constexpr int kDecodeStages = 5;

template <int TN>
struct Cfg {
  static constexpr int kStageBytes = round_up(BM * BK + TN * BK, kAlign);
  // two staging buffers of [KBC][TN] activation scales + [KBC] weight scales
  static constexpr int kScaleBytes = round_up(2 * (KBC * TN + KBC) * 4, kAlign);
  static constexpr Fp8TileShape kShape{BM, TN, BK, kMisc + kScaleBytes + kAlign};
  // M <= 16 (decode): a 5-stage ring (98 KB) and at most 85 registers a
  // thread, so that two CTAs share an SM and a GEMM launched behind this one
  // streams its first weight stages while this one finishes
  static constexpr int kMax = TN == 16 ? kDecodeStages : kMaxStages;
  static constexpr int kStages = fp8_main_stages(kShape) < kMax ? fp8_main_stages(kShape) : kMax;
  static constexpr int kSmem = kStages * kStageBytes + kScaleBytes + kMisc + kAlign;
  // partial slots: as many K blocks as tensor memory holds (up to 16), so
  // the tensor core can run that far ahead of the promotion warps
  static constexpr int kSlots = (512 / TN) < 16 ? (512 / TN) : 16;
  static constexpr int kTmemCols = pow2_cols(kSlots * TN);
  static constexpr int kColsPerWarp = TN / 2;
  static_assert(kStages >= 2, "ring too shallow");
  static_assert(kSmem <= kSmemPerCta, "smem budget");
  static_assert(kSlots >= 2 && kSlots * TN <= kTmemCols && kTmemCols <= bsk::kTmemCols, "tmem budget");
};

// A CTA's piece of work: K blocks [kb0, kb1) of tile t.
struct Seg {
  int t, kb0, kb1;
};

// The CTA's segments in order; every role walks the same sequence.
template <bool kStreamK>
struct Walk {
  long long cur, end;
  int step;
  __device__ __forceinline__ Walk(const Fp8Params& p, int total, int nkb) {
    if (kStreamK) {
      const long long U = (long long)total * nkb;
      cur = (long long)blockIdx.x * U / gridDim.x;
      end = (long long)(blockIdx.x + 1) * U / gridDim.x;
      step = 0;
    } else {
      cur = blockIdx.x;
      end = total;
      step = (int)gridDim.x;
    }
  }
  __device__ __forceinline__ bool next(const Fp8Params& p, int nkb, Seg& s) {
    if (cur >= end) return false;
    if (kStreamK) {
      s.t = (int)(cur / nkb);
      s.kb0 = (int)(cur % nkb);
      s.kb1 = (int)min((long long)nkb, s.kb0 + (end - cur));
      cur += s.kb1 - s.kb0;
    } else {
      s.t = (int)cur;
      s.kb0 = 0;
      s.kb1 = nkb;
      cur += step;
    }
    return true;
  }
};

// CTA whose stream-K range holds unit u (ranges [c U / G, (c + 1) U / G)).
__device__ __forceinline__ int sk_owner(long long u, long long U, int G) { return (int)(((u + 1) * G - 1) / U); }

// kMulti: G products Y_g = X W_g^T that share the token operand run as one
// list of tiles, product-major (tile t is tile t mod T of product t / T, T =
// tiles of one product), so a decode step's projections stream their weights
// through one grid and pay its launch, first loads and fix-ups once.
template <int TN, bool kStreamK, bool kRowwise, bool kMulti>
__global__ void __launch_bounds__(kThreads, TN == 16 ? 2 : 1)
    fp8_gemm_kernel(const __grid_constant__ typename WArg<kMulti>::type tmW,
                    const __grid_constant__ CUtensorMap tmX, const Fp8Params p) {
  static_assert(!(kMulti && kRowwise), "the multi-weight kernel is block-scaled");
  using C = Cfg<TN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + kAlign - 1) &
                                             ~static_cast<uintptr_t>(kAlign - 1));
  uint8_t* stages = base;
  float* ssa = reinterpret_cast<float*>(base + C::kStages * C::kStageBytes);  // [2][KBC][TN]
  float* ssb = ssa + 2 * KBC * TN;                                            // [2][KBC]
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::kStages * C::kStageBytes + C::kScaleBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::kStages;
  uint64_t* pfull = bars + 2 * C::kStages;     // [kSlots] partial slot written by the tensor core
  uint64_t* pempty = pfull + C::kSlots;        // [kSlots] partial slot read by the epilogue
  uint64_t* drain = pfull + 2 * C::kSlots;
  uint32_t* tmem_base = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_i = reinterpret_cast<int*>(tmem_base + 1);
  int* fix_flag = abort_i + 1;                 // stream-K: this CTA finishes the tile
  volatile int* abort_flag = abort_i;
  const WaitGuard wg{abort_flag, p.status, p.wait_ns};
  const int warp = warp_bcast((int)(threadIdx.x / 32)), lane = threadIdx.x % 32;

  // Prologue.  The producer (warp 0) initialises the barriers itself and
  // starts loading at once; it signals named barrier 2 without waiting, so the
  // tensor-memory allocation (warp 1) overlaps its first loads.  The other
  // warps wait on barrier 2 for both the barriers and the allocation.
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

  const int n_wblk = (p.N + BM - 1) / BM;
  const int n_tblk = (p.M + TN - 1) / TN;
  const int per = n_wblk * n_tblk;              // tiles of one product
  const int total = (kMulti ? p.G : 1) * per;
  const int nkb = p.K / BK;
  // tile t: product, weight-row block, token block
  auto t_g = [&](int t) { return kMulti ? t / per : 0; };
  auto t_w = [&](int t) { return (kMulti ? t % per : t) % n_wblk; };
  auto t_tok = [&](int t) { return (kMulti ? t % per : t) / n_wblk; };
  auto wmap = [&](int g) -> const CUtensorMap* {
    if constexpr (kMulti) return &tmW.m[g];
    else return &tmW;
  };

  // The producer and the MMA issuer run with the whole warp: lane 0 waits on
  // the barriers (result broadcast), one elected lane issues.
  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    PipeState<C::kStages> ps;
    uint32_t issued_mask = 0, last_phase = 0;
    bool ok = true;
    const int pre = p.pre_b < C::kStages ? p.pre_b : C::kStages;
    int item = 0;
    // The token tiles of the first `issued` items, issued once the preceding
    // kernel (the activation quantizer) has finished.  Those items sit in
    // ring slots 0 .. issued-1 of the fresh ring.
    auto late_token_loads = [&](int issued) {
      griddep_wait();
      Walk<kStreamK> w2(p, total, nkb);
      Seg s2;
      int i = 0;
      while (i < issued && w2.next(p, nkb, s2))
        for (int kb = s2.kb0; kb < s2.kb1 && i < issued; ++kb, ++i)
          if (elect_one())
            tma_load_2d(stages + i * C::kStageBytes + BM * BK, &tmX, &full[i], kb * BK, t_tok(s2.t) * TN);
      __syncwarp();
    };
    if (pre == 0) griddep_wait();
    Walk<kStreamK> w(p, total, nkb);
    Seg sg;
    while (ok && w.next(p, nkb, sg)) {
      const int wb = t_w(sg.t), tb = t_tok(sg.t);
      const CUtensorMap* mw = wmap(t_g(sg.t));
      for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
        if (!mbar_wait_warp(&empty[ps.index], ps.phase ^ 1u, wg, 50)) { ok = false; break; }
        uint8_t* st = stages + ps.index * C::kStageBytes;
        if (elect_one()) {
          mbar_arrive_expect_tx(&full[ps.index], (uint32_t)(BM * BK + TN * BK));
          tma_load_2d(st, mw, &full[ps.index], kb * BK, wb * BM);
          if (item >= pre) tma_load_2d(st + BM * BK, &tmX, &full[ps.index], kb * BK, tb * TN);
        }
        __syncwarp();
        issued_mask |= 1u << ps.index;
        last_phase = (last_phase & ~(1u << ps.index)) | (ps.phase << ps.index);
        ps.advance();
        if (++item == pre) late_token_loads(pre);
      }
    }
    if (item < pre) late_token_loads(item);   // fewer items than early weight loads (or an abort)
    if (lane == 0) {
      // copies already in flight land before the CTA can exit
      for (int s = 0; s < C::kStages; ++s)
        if (issued_mask & (1u << s)) mbar_drain(&full[s], (last_phase >> s) & 1u, 100000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // Descriptors are built once for stage 0 and advanced by byte offset / 16.
    PipeState<C::kStages> ps;
    PipeState<C::kSlots> sl;  // partial slot ring
    constexpr uint32_t idesc = idesc_e4m3(BM, TN);
    const uint64_t dW = smem_desc(smem_u32(stages), 16, 1024, kLayoutSw128);
    const uint64_t dX = smem_desc(smem_u32(stages + BM * BK), 16, 1024, kLayoutSw128);
    bool ok = true;
    Walk<kStreamK> w(p, total, nkb);
    Seg sg;
    while (ok && w.next(p, nkb, sg)) {
      if constexpr (kRowwise) {
        // W8A8: the segment's K blocks accumulate into one slot, handed to the
        // epilogue once
        if (!mbar_wait_warp(&pempty[sl.index], sl.phase ^ 1u, wg, 62)) { ok = false; break; }
        const uint32_t d = tmem + sl.index * TN;
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          if (!mbar_wait_warp(&full[ps.index], ps.phase, wg, 63)) { ok = false; break; }
          tc_fence_after();
          const uint64_t so = (uint64_t)((ps.index * C::kStageBytes) >> 4);
          if (elect_one()) {
#pragma unroll
            for (int j = 0; j < BK / 32; ++j)
              mma_e4m3(d, dW + so + 2 * j, dX + so + 2 * j, idesc, (kb > sg.kb0 || j > 0) ? 1u : 0u);
            tc_commit(&empty[ps.index]);
          }
          __syncwarp();
          ps.advance();
        }
        if (!ok) break;
        if (elect_one()) tc_commit(&pfull[sl.index]);
        __syncwarp();
        sl.advance();
      } else {
      for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
        if (!mbar_wait_warp(&pempty[sl.index], sl.phase ^ 1u, wg, 60)) { ok = false; break; }
        if (!mbar_wait_warp(&full[ps.index], ps.phase, wg, 61)) { ok = false; break; }
        tc_fence_after();
        const uint64_t so = (uint64_t)((ps.index * C::kStageBytes) >> 4);
        const uint32_t d = tmem + sl.index * TN;
        if (elect_one()) {
#pragma unroll
          for (int j = 0; j < BK / 32; ++j)
            mma_e4m3(d, dW + so + 2 * j, dX + so + 2 * j, idesc, j > 0 ? 1u : 0u);  // 32 B of K per MMA
          tc_commit(&empty[ps.index]);
          tc_commit(&pfull[sl.index]);
        }
        __syncwarp();
        ps.advance();
        sl.advance();
      }
      }
    }
    if (elect_one()) {
      tc_commit(drain);
      mbar_drain(drain, 0, 1000000000ull);
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------------ promotion + epilogue
    // Walks (segment, chunk of KBC K blocks) in order.  The scales of the next
    // chunk are staged into shared memory with cp.async while this chunk is
    // promoted, so no K block waits on a global load.  Every epilogue warp runs
    // the same sequence of named barriers; after an abort the warps keep
    // walking (skipping the waits and the work) so the barriers still match,
    // and stream-K tiles are still counted in so the counters return to zero.
    constexpr int NC = C::kColsPerWarp;
    const int q = warp % 4, half = (warp - kEpiWarp0) / 4;
    const int col0 = half * NC;
    const int r = q * 32 + lane;                     // weight row within the tile
    const int etid = threadIdx.x - kEpiWarp0 * 32;  // 0 .. 255
    griddep_wait();                                 // activation scales come from the preceding kernel
    PipeState<C::kSlots> sl;
    bool ok = true;
    auto nchunks = [&](const Seg& s) { return (s.kb1 - s.kb0 + KBC - 1) / KBC; };
    auto stage_scales = [&](const Seg& s, int c, int buf) {
      const int wb = t_w(s.t), tb = t_tok(s.t);
      const float* sfb = kMulti ? pick(p.sfb_g, t_g(s.t)) : p.sfb;
      float* da = ssa + buf * KBC * TN;
      float* db = ssb + buf * KBC;
      for (int i = etid; i < KBC * TN; i += 256) {
        const int kbl = i / TN, m = i % TN;
        const int kb = s.kb0 + c * KBC + kbl, ma = tb * TN + m;
        const bool valid = kb < s.kb1 && ma < p.M;
        const float* src = valid ? p.sfa + (size_t)kb * p.M + ma : p.sfa;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(da + i)), "l"(src),
                     "r"(valid ? 4 : 0)
                     : "memory");
      }
      for (int i = etid; i < KBC; i += 256) {
        const int kb = s.kb0 + c * KBC + i;
        const bool valid = kb < s.kb1;
        const float* src = valid ? sfb + (size_t)wb * nkb + kb : sfb;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(db + i)), "l"(src),
                     "r"(valid ? 4 : 0)
                     : "memory");
      }
    };
    auto store_out = [&](const Seg& s, const float (&y)[NC]) {
      const int n = t_w(s.t) * BM + r;                  // weight row = output column
      const int m0 = t_tok(s.t) * TN + col0;            // first token of this warp's columns
      void* const out = kMulti ? pick(p.out_g, t_g(s.t)) : p.out;
      if (n >= p.N) return;
      const float sw = kRowwise ? __ldg(p.sfb + n) : 1.0f;   // W8A8: channel scale of this row
#pragma unroll
      for (int i = 0; i < NC; ++i) {
        const int m = m0 + i;
        if (m < p.M) {
          const float v = kRowwise ? y[i] * (__ldg(p.sfa + m) * sw) : y[i];
          if (p.out_bf16)
            reinterpret_cast<__nv_bfloat16*>(out)[(size_t)m * p.ldo + n] = __float2bfloat16_rn(v);
          else
            reinterpret_cast<float*>(out)[(size_t)m * p.ldo + n] = v;
        }
      }
    };
    // End of a segment: a whole tile is stored; a stream-K piece goes to the
    // workspace and the last of the tile's CTAs sums the pieces (in K order)
    // and stores them.  Every epilogue warp takes part (named barrier 1).
    // acc is reset for the next segment.
    auto finish = [&](const Seg& sg, float (&acc)[NC], bool ok) {
      if (!kStreamK || (sg.kb0 == 0 && sg.kb1 == nkb)) {
        if (ok) store_out(sg, acc);
      } else {
        // stream-K piece of a tile: partial to the workspace, count in; the
        // last of the tile's CTAs sums the pieces in K order
        const long long U = (long long)total * nkb, u0 = (long long)sg.t * nkb;
        const int c_first = sk_owner(u0, U, (int)gridDim.x);
        const int n_parts = sk_owner(u0 + nkb - 1, U, (int)gridDim.x) - c_first + 1;
        const int j = (int)blockIdx.x - c_first;
        float* parts = p.work + (size_t)sg.t * p.maxc * (BM * TN);
        float4* mine = reinterpret_cast<float4*>(parts + (size_t)j * (BM * TN) + r * TN + col0);
#pragma unroll
        for (int i = 0; i < NC; i += 4) mine[i / 4] = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
        // One thread counts the CTA in with an acquire-release add: the
        // barrier orders every thread's partial before its release, and if
        // it is the last piece its acquire (passed on by the second barrier)
        // orders the other CTAs' partials before the reads below.
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (etid == 0) {
          int old;
          asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(p.counters + sg.t) : "memory");
          *fix_flag = old == n_parts - 1;
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (*fix_flag) {
          // every piece, this CTA's own included, summed from the workspace
          // (L2) in K order
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
      }
#pragma unroll
      for (int i = 0; i < NC; ++i) acc[i] = 0.0f;
    };
    if constexpr (kRowwise) {
      // W8A8: one accumulator per segment, scaled once at the store
      Walk<kStreamK> w(p, total, nkb);
      Seg sg;
      float acc[NC];
#pragma unroll
      for (int i = 0; i < NC; ++i) acc[i] = 0.0f;
      while (w.next(p, nkb, sg)) {
        if (ok) {
          int w_ok = 1;
          if (lane == 0) w_ok = mbar_wait(&pfull[sl.index], sl.phase, wg, 72) ? 1 : 0;
          ok = __shfl_sync(0xffffffffu, w_ok, 0) != 0;
        }
        if (ok) {
          tc_fence_after();
          constexpr int CH = NC < 32 ? NC : 32;
#pragma unroll
          for (int c0 = 0; c0 < NC; c0 += CH) {
            uint32_t v[CH];
            tmem_ld_cols<CH>(tmem + ((uint32_t)(q * 32) << 16) + sl.index * TN + col0 + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < CH; ++i) acc[c0 + i] = __uint_as_float(v[i]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&pempty[sl.index]);
        }
        sl.advance();
        finish(sg, acc, ok);
      }
    } else {
    Walk<kStreamK> w(p, total, nkb);
    Seg sg;
    bool have = w.next(p, nkb, sg);
    int c = 0, qi = 0;
    if (have) stage_scales(sg, 0, 0);
    asm volatile("cp.async.commit_group;" ::: "memory");
    float acc[NC];
#pragma unroll
    for (int i = 0; i < NC; ++i) acc[i] = 0.0f;
    while (have) {
      Seg sn = sg;
      int cn = c + 1;
      bool haven = true;
      if (cn == nchunks(sg)) {
        cn = 0;
        haven = w.next(p, nkb, sn);
      }
      if (haven) stage_scales(sn, cn, (qi + 1) & 1);
      asm volatile("cp.async.commit_group;" ::: "memory");
      asm volatile("cp.async.wait_group 1;" ::: "memory");
      asm volatile("bar.sync 1, 256;" ::: "memory");
      {
        // fold the weight block scale into the token scales once per chunk:
        // csa[kb][m] = sb[kb] * sa[kb][m], the same factor for every row
        float* wsa = ssa + (qi & 1) * KBC * TN;
        const float* wsb = ssb + (qi & 1) * KBC;
        for (int i = etid; i < KBC * TN; i += 256) wsa[i] *= wsb[i / TN];
        asm volatile("bar.sync 1, 256;" ::: "memory");
      }
      const float* csa = ssa + (qi & 1) * KBC * TN;
      const int kc0 = sg.kb0 + c * KBC;                // first K block of the chunk
      const int kb_end = min(sg.kb1, kc0 + KBC);
      // Small tiles fold G partial slots per round trip (wait all, load all,
      // one tcgen05.wait::ld, release all) so the latency of the hand-off is
      // paid once per G K blocks.
      constexpr int kFold = TN == 16 ? 16 : 64;   // registers for the folded slots (two CTAs per SM at TN 16)
      constexpr int G = NC <= 32 ? (kFold / NC < 8 ? kFold / NC : 8) : 1;
      int kb = kc0;
      if constexpr (G > 1) {
        for (; kb + G <= kb_end; kb += G) {
          uint32_t idx[G];
#pragma unroll
          for (int i = 0; i < G; ++i) {
            idx[i] = sl.index;
            if (ok) {
              int w_ok = 1;
              if (lane == 0) w_ok = mbar_wait(&pfull[sl.index], sl.phase, wg, 71) ? 1 : 0;
              w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
              ok = w_ok != 0;
            }
            sl.advance();
          }
          if (ok) {
            tc_fence_after();
            uint32_t v[G][NC];
#pragma unroll
            for (int i = 0; i < G; ++i)
              tmem_ld_cols<NC>(tmem + ((uint32_t)(q * 32) << 16) + idx[i] * TN + col0, v[i]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
#pragma unroll
              for (int i = 0; i < G; ++i) mbar_arrive(&pempty[idx[i]]);
            }
#pragma unroll
            for (int i = 0; i < G; ++i) {
              const float4* s4 = reinterpret_cast<const float4*>(csa + (kb + i - kc0) * TN + col0);
#pragma unroll
              for (int j = 0; j < NC; j += 4) {
                const float4 sc = s4[j / 4];  // same address in every lane: one broadcast
                acc[j] = fmaf(__uint_as_float(v[i][j]), sc.x, acc[j]);
                acc[j + 1] = fmaf(__uint_as_float(v[i][j + 1]), sc.y, acc[j + 1]);
                acc[j + 2] = fmaf(__uint_as_float(v[i][j + 2]), sc.z, acc[j + 2]);
                acc[j + 3] = fmaf(__uint_as_float(v[i][j + 3]), sc.w, acc[j + 3]);
              }
            }
          }
        }
      }
      for (; kb < kb_end; ++kb) {
        if (ok) {
          int w_ok = 1;
          if (lane == 0) w_ok = mbar_wait(&pfull[sl.index], sl.phase, wg, 70) ? 1 : 0;
          w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
          ok = w_ok != 0;
        }
        if (ok) {
          tc_fence_after();
          const float4* s4 = reinterpret_cast<const float4*>(csa + (kb - kc0) * TN + col0);
          if constexpr (!kStreamK) {
            // the warp's whole slot in registers with one wait, the slot handed
            // back, then the fold (two columns per packed FMA)
            uint32_t v[NC];
            tmem_ld_cols<NC>(tmem + ((uint32_t)(q * 32) << 16) + sl.index * TN + col0, v);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&pempty[sl.index]);
#pragma unroll
            for (int i = 0; i < NC; i += 4) {
              const float4 sc = s4[i / 4];
              const float2 lo = __ffma2_rn(make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])),
                                           make_float2(sc.x, sc.y), make_float2(acc[i], acc[i + 1]));
              const float2 hi = __ffma2_rn(make_float2(__uint_as_float(v[i + 2]), __uint_as_float(v[i + 3])),
                                           make_float2(sc.z, sc.w), make_float2(acc[i + 2], acc[i + 3]));
              acc[i] = lo.x;
              acc[i + 1] = lo.y;
              acc[i + 2] = hi.x;
              acc[i + 3] = hi.y;
            }
          } else {
            // stream-K (registers also hold the fix-up): two halves, one wait each
            constexpr int CH = NC < 32 ? NC : 32;
#pragma unroll
            for (int c0 = 0; c0 < NC; c0 += CH) {
              uint32_t v[CH];
              tmem_ld_cols<CH>(tmem + ((uint32_t)(q * 32) << 16) + sl.index * TN + col0 + c0, v);
              tmem_ld_wait();
              if (c0 + CH == NC) {
                // every column of the slot is in registers: hand the slot back
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&pempty[sl.index]);
              }
#pragma unroll
              for (int i = 0; i < CH; i += 4) {
                const float4 sc = s4[(c0 + i) / 4];
                acc[c0 + i] = fmaf(__uint_as_float(v[i]), sc.x, acc[c0 + i]);
                acc[c0 + i + 1] = fmaf(__uint_as_float(v[i + 1]), sc.y, acc[c0 + i + 1]);
                acc[c0 + i + 2] = fmaf(__uint_as_float(v[i + 2]), sc.z, acc[c0 + i + 2]);
                acc[c0 + i + 3] = fmaf(__uint_as_float(v[i + 3]), sc.w, acc[c0 + i + 3]);
              }
            }
          }
        }
        sl.advance();
      }
      if (cn == 0) finish(sg, acc, ok);  // the segment's last chunk
      asm volatile("bar.sync 1, 256;" ::: "memory");  // this buffer may be refilled next iteration
      sg = sn;
      c = cn;
      have = haven;
      ++qi;
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
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

template <int TN, bool kStreamK, bool kRowwise, bool kMulti = false>
static cudaError_t launch_tn(const Fp8Launch& L, cudaStream_t stream) {
  using C = Cfg<TN>;
  auto kern = fp8_gemm_kernel<TN, kStreamK, kRowwise, kMulti>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  // all of the SM's unified memory as shared memory, so two decode CTAs fit
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  if constexpr (kMulti)
    return launch_kernel(kern, (unsigned)L.grid, kThreads, (size_t)C::kSmem, stream, 1, L.tmA_g, L.tmB, L.p);
  else
    return launch_kernel(kern, (unsigned)L.grid, kThreads, (size_t)C::kSmem, stream, 1, L.tmA, L.tmB, L.p);
}

}  // namespace fp8

int fp8_tile_n(long long M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  return 128;
}

int fp8_stages(int tile_n) {
  switch (tile_n) {
    case 16: return fp8::Cfg<16>::kStages;
    case 32: return fp8::Cfg<32>::kStages;
    case 64: return fp8::Cfg<64>::kStages;
    case 128: return fp8::Cfg<128>::kStages;
  }
  return 0;
}

template <bool kStreamK, bool kRowwise>
static cudaError_t launch_sk(const Fp8Launch& L, cudaStream_t stream) {
  switch (L.tile_n) {
    case 16: return fp8::launch_tn<16, kStreamK, kRowwise>(L, stream);
    case 32: return fp8::launch_tn<32, kStreamK, kRowwise>(L, stream);
    case 64: return fp8::launch_tn<64, kStreamK, kRowwise>(L, stream);
    case 128: return fp8::launch_tn<128, kStreamK, kRowwise>(L, stream);
  }
  return cudaErrorInvalidValue;
}

// Multi-weight launches: block-scaled, decode tiles (M <= 32) only.
template <bool kStreamK>
static cudaError_t launch_multi(const Fp8Launch& L, cudaStream_t stream) {
  switch (L.tile_n) {
    case 16: return fp8::launch_tn<16, kStreamK, false, true>(L, stream);
    case 32: return fp8::launch_tn<32, kStreamK, false, true>(L, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_fp8_gemm(const Fp8Launch& L, cudaStream_t stream) {
  if (L.grid <= 0) return cudaErrorInvalidValue;
  if (L.p.G > 1) {
    if (L.p.G > kMaxProducts || L.p.rowwise) return cudaErrorInvalidValue;
    return L.p.stream_k ? launch_multi<true>(L, stream) : launch_multi<false>(L, stream);
  }
  if (L.p.rowwise) return L.p.stream_k ? launch_sk<true, true>(L, stream) : launch_sk<false, true>(L, stream);
  return L.p.stream_k ? launch_sk<true, false>(L, stream) : launch_sk<false, false>(L, stream);
}

}  // namespace bsk
