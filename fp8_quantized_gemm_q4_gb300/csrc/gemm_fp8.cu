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
// One persistent CTA per SM walks (weight block, token block) tiles.
//   warp 0      TMA producer: weight tile [128 x 128] + token tile [TN x 128]
//   warp 1      tensor-memory allocator, single-lane MMA issuer
//               (tcgen05.mma kind::f8f6f4, K = 32 per instruction)
//   warps 4-11  promotion / epilogue: two warps per 32-lane quarter, each
//               owning half of the TN token columns of its weight rows
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

template <int TN, int kSplit>
struct Cfg {
  static constexpr int kStageBytes = round_up(BM * BK + TN * BK, kAlign);
  // two staging buffers of [KBC][TN] activation scales + [KBC] weight scales
  static constexpr int kScaleBytes = round_up(2 * (KBC * TN + KBC) * 4, kAlign);
  // split-K partner's partial sums [BM rows][TN], written through DSMEM
  // (split mode only: elsewhere the bytes go to the stage ring)
  static constexpr int kRedBytes = kSplit > 1 ? round_up(BM * TN * 4, kAlign) : 0;
  static constexpr Fp8TileShape kShape{BM, TN, BK, kMisc + kScaleBytes + kRedBytes + kAlign};
  static constexpr int kStages = fp8_main_stages(kShape) < kMaxStages ? fp8_main_stages(kShape) : kMaxStages;
  static constexpr int kSmem = kStages * kStageBytes + kScaleBytes + kRedBytes + kMisc + kAlign;
  // partial slots: as many K blocks as tensor memory holds (up to 16), so
  // the tensor core can run that far ahead of the promotion warps
  static constexpr int kSlots = (512 / TN) < 16 ? (512 / TN) : 16;
  static constexpr int kTmemCols = pow2_cols(kSlots * TN);
  static constexpr int kColsPerWarp = TN / 2;
  static_assert(kStages >= 2, "ring too shallow");
  static_assert(kSmem <= kSmemPerCta, "smem budget");
  static_assert(kSlots >= 2 && kSlots * TN <= kTmemCols && kTmemCols <= bsk::kTmemCols, "tmem budget");
};

// kSplit == 2: a cluster of two CTAs shares one tile, each streaming half of
// the K blocks; the peer's fp32 partials reach the leader through distributed
// shared memory at the end (decode shapes: twice as many SMs pull weights).
template <int TN, int kSplit>
__global__ void __launch_bounds__(kThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                    const Fp8Params p) {
  using C = Cfg<TN, kSplit>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + kAlign - 1) &
                                             ~static_cast<uintptr_t>(kAlign - 1));
  uint8_t* stages = base;
  float* ssa = reinterpret_cast<float*>(base + C::kStages * C::kStageBytes);  // [2][KBC][TN]
  float* ssb = ssa + 2 * KBC * TN;                                            // [2][KBC]
  float* red = reinterpret_cast<float*>(base + C::kStages * C::kStageBytes + C::kScaleBytes);  // [BM][TN]
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(base + C::kStages * C::kStageBytes + C::kScaleBytes + C::kRedBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::kStages;
  uint64_t* pfull = bars + 2 * C::kStages;     // [kSlots] partial slot written by the tensor core
  uint64_t* pempty = pfull + C::kSlots;        // [kSlots] partial slot read by the epilogue
  uint64_t* drain = pfull + 2 * C::kSlots;
  uint32_t* tmem_base = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_i = reinterpret_cast<int*>(tmem_base + 1);
  volatile int* abort_flag = abort_i;
  const WaitGuard wg{abort_flag, p.status, p.wait_ns};
  const int warp = warp_bcast((int)(threadIdx.x / 32)), lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
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
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmX);
  }
  if (warp == 1) {
    tmem_alloc(tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = warp_bcast(*tmem_base);

  const int n_wblk = (p.N + BM - 1) / BM;
  const int n_tblk = (p.M + TN - 1) / TN;
  const int total = n_wblk * n_tblk;
  const int nkb_all = p.K / BK;
  // split mode: this CTA's K blocks [kb0, kb0 + nkb); tiles are walked per cluster
  const uint32_t srank = kSplit > 1 ? warp_bcast(cluster_ctarank()) : 0u;
  const int kb0 = kSplit > 1 ? (int)srank * ((nkb_all + 1) / 2) : 0;
  const int nkb = kSplit > 1 ? (srank == 0 ? (nkb_all + 1) / 2 : nkb_all / 2) : nkb_all;
  const int t_first = kSplit > 1 ? (int)blockIdx.x / 2 : (int)blockIdx.x;
  const int t_step = kSplit > 1 ? (int)gridDim.x / 2 : (int)gridDim.x;

  // split mode: the tile's partial sums of this thread, kept for the exchange
  float facc[C::kColsPerWarp];
  int f_n = 0, f_m0 = 0;
  bool f_have = false;
#pragma unroll
  for (int i = 0; i < C::kColsPerWarp; ++i) facc[i] = 0.0f;

  // The producer and the MMA issuer run with the whole warp: lane 0 waits on
  // the barriers (result broadcast), one elected lane issues.
  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    PipeState<C::kStages> ps;
    uint32_t issued_mask = 0, last_phase = 0;
    bool ok = true;
    for (int t = t_first; t < total && ok; t += t_step) {
      const int wb = t % n_wblk, tb = t / n_wblk;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait_warp(&empty[ps.index], ps.phase ^ 1u, wg, 50)) { ok = false; break; }
        uint8_t* st = stages + ps.index * C::kStageBytes;
        if (elect_one()) {
          mbar_arrive_expect_tx(&full[ps.index], (uint32_t)(BM * BK + TN * BK));
          tma_load_2d(st, &tmW, &full[ps.index], (kb0 + kb) * BK, wb * BM);
          tma_load_2d(st + BM * BK, &tmX, &full[ps.index], (kb0 + kb) * BK, tb * TN);
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
    // Descriptors are built once for stage 0 and advanced by byte offset / 16.
    PipeState<C::kStages> ps;
    PipeState<C::kSlots> sl;  // partial slot ring
    constexpr uint32_t idesc = idesc_e4m3(BM, TN);
    const uint64_t dW = smem_desc(smem_u32(stages), 16, 1024, kLayoutSw128);
    const uint64_t dX = smem_desc(smem_u32(stages + BM * BK), 16, 1024, kLayoutSw128);
    bool ok = true;
    for (int t = t_first; t < total && ok; t += t_step) {
      for (int kb = 0; kb < nkb; ++kb) {
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
    if (elect_one()) {
      tc_commit(drain);
      mbar_drain(drain, 0, 1000000000ull);
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------------ promotion + epilogue
    // Walks (tile, chunk of KBC K blocks) in order.  The scales of the next
    // chunk are staged into shared memory with cp.async while this chunk is
    // promoted, so no K block waits on a global load.  Every epilogue warp runs
    // the same sequence of named barriers; after an abort the warps keep
    // walking (skipping the waits and the work) so the barriers still match.
    constexpr int NC = C::kColsPerWarp;
    const int q = warp % 4, half = (warp - kEpiWarp0) / 4;
    const int col0 = half * NC;
    const int etid = threadIdx.x - kEpiWarp0 * 32;  // 0 .. 255
    const int nchunk = (nkb + KBC - 1) / KBC;
    PipeState<C::kSlots> sl;
    bool ok = true;
    auto stage_scales = [&](int t, int c, int buf) {
      const int wb = t % n_wblk, tb = t / n_wblk;
      float* da = ssa + buf * KBC * TN;
      float* db = ssb + buf * KBC;
      for (int i = etid; i < KBC * TN; i += 256) {
        const int kbl = i / TN, m = i % TN;
        const int kb = c * KBC + kbl, ma = tb * TN + m;
        const bool valid = kb < nkb && ma < p.M;
        const float* src = valid ? p.sfa + (size_t)(kb0 + kb) * p.M + ma : p.sfa;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(da + i)), "l"(src),
                     "r"(valid ? 4 : 0)
                     : "memory");
      }
      for (int i = etid; i < KBC; i += 256) {
        const int kb = c * KBC + i;
        const bool valid = kb < nkb;
        const float* src = valid ? p.sfb + (size_t)wb * nkb_all + kb0 + kb : p.sfb;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(db + i)), "l"(src),
                     "r"(valid ? 4 : 0)
                     : "memory");
      }
    };
    int t = t_first, c = 0, qi = 0;
    if (t < total) stage_scales(t, 0, 0);
    asm volatile("cp.async.commit_group;" ::: "memory");
    float acc[NC];
#pragma unroll
    for (int i = 0; i < NC; ++i) acc[i] = 0.0f;
    while (t < total) {
      int tn = t, cn = c + 1;
      if (cn == nchunk) {
        cn = 0;
        tn = t + t_step;
      }
      if (tn < total) stage_scales(tn, cn, (qi + 1) & 1);
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
      const int wb = t % n_wblk, tb = t / n_wblk;
      const int n = wb * BM + q * 32 + lane;            // weight row = output column
      const int m0 = tb * TN + col0;                    // first token of this warp's columns
      const int kb_end = min(nkb, (c + 1) * KBC);
      // Small tiles fold G partial slots per round trip (wait all, load all,
      // one tcgen05.wait::ld, release all) so the latency of the hand-off is
      // paid once per G K blocks.
      constexpr int G = NC <= 32 ? (64 / NC < 8 ? 64 / NC : 8) : 1;
      int kb = c * KBC;
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
              const float4* s4 = reinterpret_cast<const float4*>(csa + (kb + i - c * KBC) * TN + col0);
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
          const float4* s4 = reinterpret_cast<const float4*>(csa + (kb - c * KBC) * TN + col0);
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
        sl.advance();
      }
      if (cn == 0 && kSplit > 1) {
        // split mode (one tile per cluster): keep the partial for the exchange
#pragma unroll
        for (int i = 0; i < NC; ++i) facc[i] = acc[i];
        f_n = n;
        f_m0 = m0;
        f_have = ok;
      } else if (cn == 0) {
        // the tile's last chunk: write it and reset the accumulators
        if (ok && n < p.N) {
#pragma unroll
          for (int i = 0; i < NC; ++i) {
            const int m = m0 + i;
            if (m < p.M) {
              if (p.out_bf16)
                reinterpret_cast<__nv_bfloat16*>(p.out)[(size_t)m * p.ldo + n] = __float2bfloat16_rn(acc[i]);
              else
                reinterpret_cast<float*>(p.out)[(size_t)m * p.ldo + n] = acc[i];
            }
          }
        }
#pragma unroll
        for (int i = 0; i < NC; ++i) acc[i] = 0.0f;
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");  // this buffer may be refilled next iteration
      t = tn;
      c = cn;
      ++qi;
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    if (kSplit > 1 && srank == 1 && f_have) {
      // hand the partial sums to the leader's reduction buffer (DSMEM)
      const uint32_t dst = mapa_shared(smem_u32(red + (q * 32 + lane) * TN + col0), 0);
#pragma unroll
      for (int i = 0; i < NC; ++i)
        asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dst + 4 * i), "f"(facc[i]) : "memory");
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (kSplit > 1) {
    cluster_sync();  // the peer's partials have landed in the leader's buffer
    if (srank == 0 && warp >= kEpiWarp0 && f_have && f_n < p.N) {
      const int q = warp % 4, col0 = ((warp - kEpiWarp0) / 4) * C::kColsPerWarp;
      const float* other = red + (q * 32 + lane) * TN + col0;
#pragma unroll
      for (int i = 0; i < C::kColsPerWarp; ++i) {
        const int m = f_m0 + i;
        const float y = facc[i] + (nkb_all > 1 ? other[i] : 0.0f);
        if (m < p.M) {
          if (p.out_bf16)
            reinterpret_cast<__nv_bfloat16*>(p.out)[(size_t)m * p.ldo + f_n] = __float2bfloat16_rn(y);
          else
            reinterpret_cast<float*>(p.out)[(size_t)m * p.ldo + f_n] = y;
        }
      }
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int TN, int kSplit>
static cudaError_t launch_tn(const Fp8Launch& L, cudaStream_t stream) {
  using C = Cfg<TN, kSplit>;
  auto kern = fp8_gemm_kernel<TN, kSplit>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  if (kSplit == 1) {
    kern<<<L.grid, kThreads, C::kSmem, stream>>>(L.tmA, L.tmB, L.p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)L.grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, L.tmA, L.tmB, L.p);
}

}  // namespace fp8

int fp8_tile_n(long long M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  return 128;
}

cudaError_t launch_fp8_gemm(const Fp8Launch& L, cudaStream_t stream) {
  if (L.p.splits == 2) {
    if (L.grid <= 0 || (L.grid & 1)) return cudaErrorInvalidValue;
    switch (L.tile_n) {
      case 16: return fp8::launch_tn<16, 2>(L, stream);
      case 32: return fp8::launch_tn<32, 2>(L, stream);
    }
    return cudaErrorInvalidValue;
  }
  switch (L.tile_n) {
    case 16: return fp8::launch_tn<16, 1>(L, stream);
    case 32: return fp8::launch_tn<32, 1>(L, stream);
    case 64: return fp8::launch_tn<64, 1>(L, stream);
    case 128: return fp8::launch_tn<128, 1>(L, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace bsk
