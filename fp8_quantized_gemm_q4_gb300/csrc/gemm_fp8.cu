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
// the block's partial product into one of two tensor-memory slots and the
// epilogue warps fold it into fp32 registers, acc += partial * sb * sa, while
// the tensor core fills the other slot.
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

template <int TN>
struct Cfg {
  static constexpr int kStageBytes = round_up(BM * BK + TN * BK, kAlign);
  // two staging buffers of [KBC][TN] activation scales + [KBC] weight scales
  static constexpr int kScaleBytes = round_up(2 * (KBC * TN + KBC) * 4, kAlign);
  static constexpr Fp8TileShape kShape{BM, TN, BK, kMisc + kScaleBytes + kAlign};
  static constexpr int kStages = fp8_main_stages(kShape) < kMaxStages ? fp8_main_stages(kShape) : kMaxStages;
  static constexpr int kSmem = kStages * kStageBytes + kScaleBytes + kMisc + kAlign;
  static constexpr int kTmemCols = pow2_cols(2 * TN);
  static constexpr int kColsPerWarp = TN / 2;
  static_assert(kStages >= 2, "ring too shallow");
  static_assert(kSmem <= kSmemPerCta, "smem budget");
  static_assert(2 * TN <= kTmemCols && kTmemCols <= bsk::kTmemCols, "tmem budget");
};

template <int TN>
__global__ void __launch_bounds__(kThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                    const Fp8Params p) {
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
  uint64_t* pfull = bars + 2 * C::kStages;     // [2] partial slot written by the tensor core
  uint64_t* pempty = pfull + 2;                // [2] partial slot read by the epilogue
  uint64_t* drain = pfull + 4;
  uint32_t* tmem_base = reinterpret_cast<uint32_t*>(pfull + 5);
  int* abort_i = reinterpret_cast<int*>(tmem_base + 1);
  volatile int* abort_flag = abort_i;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
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
  const uint32_t tmem = *tmem_base;

  const int n_wblk = (p.N + BM - 1) / BM;
  const int n_tblk = (p.M + TN - 1) / TN;
  const int total = n_wblk * n_tblk;
  const int nkb = p.K / BK;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ TMA producer
    PipeState<C::kStages> ps;
    uint32_t issued_mask = 0, last_phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const int wb = t % n_wblk, tb = t / n_wblk;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(&empty[ps.index], ps.phase ^ 1u, abort_flag, p.status, 50)) { ok = false; break; }
        uint8_t* st = stages + ps.index * C::kStageBytes;
        mbar_arrive_expect_tx(&full[ps.index], (uint32_t)(BM * BK + TN * BK));
        tma_load_2d(st, &tmW, &full[ps.index], kb * BK, wb * BM);
        tma_load_2d(st + BM * BK, &tmX, &full[ps.index], kb * BK, tb * TN);
        issued_mask |= 1u << ps.index;
        last_phase = (last_phase & ~(1u << ps.index)) | (ps.phase << ps.index);
        ps.advance();
      }
    }
    if (*abort_flag) {
      for (int s = 0; s < C::kStages; ++s)
        if (issued_mask & (1u << s)) {
          const uint64_t t0 = globaltimer();
          while (!mbar_try_wait(&full[s], (last_phase >> s) & 1u) && globaltimer() - t0 < 100000000ull) {
          }
        }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------------ MMA issuer
    PipeState<C::kStages> ps;
    uint32_t slot = 0, slot_phase = 0;  // partial slot ring (2 slots)
    constexpr uint32_t idesc = idesc_e4m3(BM, TN);
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(&pempty[slot], slot_phase ^ 1u, abort_flag, p.status, 60)) { ok = false; break; }
        if (!mbar_wait(&full[ps.index], ps.phase, abort_flag, p.status, 61)) { ok = false; break; }
        tc_fence_after();
        uint8_t* st = stages + ps.index * C::kStageBytes;
        const uint32_t sw = smem_u32(st), sx = smem_u32(st + BM * BK);
        const uint32_t d = tmem + slot * TN;
#pragma unroll
        for (int j = 0; j < BK / 32; ++j)
          mma_e4m3(d, smem_desc(sw + 32 * j, 16, 1024, kLayoutSw128), smem_desc(sx + 32 * j, 16, 1024, kLayoutSw128),
                   idesc, j > 0 ? 1u : 0u);
        tc_commit(&empty[ps.index]);
        tc_commit(&pfull[slot]);
        ps.advance();
        slot ^= 1u;
        if (slot == 0) slot_phase ^= 1u;
      }
    }
    tc_commit(drain);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(drain, 0) && globaltimer() - t0 < 1000000000ull) {
    }
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
    uint32_t slot = 0, slot_phase = 0;
    bool ok = true;
    auto stage_scales = [&](int t, int c, int buf) {
      const int wb = t % n_wblk, tb = t / n_wblk;
      float* da = ssa + buf * KBC * TN;
      float* db = ssb + buf * KBC;
      for (int i = etid; i < KBC * TN; i += 256) {
        const int kbl = i / TN, m = i % TN;
        const int kb = c * KBC + kbl, ma = tb * TN + m;
        const bool valid = kb < nkb && ma < p.M;
        const float* src = valid ? p.sfa + (size_t)kb * p.M + ma : p.sfa;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(da + i)), "l"(src),
                     "r"(valid ? 4 : 0)
                     : "memory");
      }
      for (int i = etid; i < KBC; i += 256) {
        const int kb = c * KBC + i;
        const bool valid = kb < nkb;
        const float* src = valid ? p.sfb + (size_t)wb * nkb + kb : p.sfb;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(db + i)), "l"(src),
                     "r"(valid ? 4 : 0)
                     : "memory");
      }
    };
    int t = blockIdx.x, c = 0, qi = 0;
    if (t < total) stage_scales(t, 0, 0);
    asm volatile("cp.async.commit_group;" ::: "memory");
    float acc[NC];
#pragma unroll
    for (int i = 0; i < NC; ++i) acc[i] = 0.0f;
    while (t < total) {
      int tn = t, cn = c + 1;
      if (cn == nchunk) {
        cn = 0;
        tn = t + gridDim.x;
      }
      if (tn < total) stage_scales(tn, cn, (qi + 1) & 1);
      asm volatile("cp.async.commit_group;" ::: "memory");
      asm volatile("cp.async.wait_group 1;" ::: "memory");
      asm volatile("bar.sync 1, 256;" ::: "memory");
      const float* csa = ssa + (qi & 1) * KBC * TN;
      const float* csb = ssb + (qi & 1) * KBC;
      const int wb = t % n_wblk, tb = t / n_wblk;
      const int n = wb * BM + q * 32 + lane;            // weight row = output column
      const int m0 = tb * TN + col0;                    // first token of this warp's columns
      const int kb_end = min(nkb, (c + 1) * KBC);
      for (int kb = c * KBC; kb < kb_end; ++kb) {
        if (ok) {
          int w_ok = 1;
          if (lane == 0) w_ok = mbar_wait(&pfull[slot], slot_phase, abort_flag, p.status, 70) ? 1 : 0;
          w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
          ok = w_ok != 0;
        }
        if (ok) {
          tc_fence_after();
          const float sbv = csb[kb - c * KBC];
          const float* sa_row = csa + (kb - c * KBC) * TN + col0;
          constexpr int CH = NC < 32 ? NC : 32;
#pragma unroll
          for (int c0 = 0; c0 < NC; c0 += CH) {
            uint32_t v[CH];
            tmem_ld_cols<CH>(tmem + ((uint32_t)(q * 32) << 16) + slot * TN + col0 + c0, v);
            tmem_ld_wait();
            if (c0 + CH == NC) {
              // every column of the slot is in registers: hand the slot back
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&pempty[slot]);
            }
#pragma unroll
            for (int i = 0; i < CH; ++i) acc[c0 + i] = fmaf(__uint_as_float(v[i]), sbv * sa_row[c0 + i], acc[c0 + i]);
          }
        }
        slot ^= 1u;
        if (slot == 0) slot_phase ^= 1u;
      }
      if (cn == 0) {
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
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int TN>
static cudaError_t launch_tn(const Fp8Launch& L, cudaStream_t stream) {
  using C = Cfg<TN>;
  auto kern = fp8_gemm_kernel<TN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<L.grid, kThreads, C::kSmem, stream>>>(L.tmA, L.tmB, L.p);
  return cudaGetLastError();
}

}  // namespace fp8

int fp8_tile_n(long long M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  return 128;
}

cudaError_t launch_fp8_gemm(const Fp8Launch& L, cudaStream_t stream) {
  switch (L.tile_n) {
    case 16: return fp8::launch_tn<16>(L, stream);
    case 32: return fp8::launch_tn<32>(L, stream);
    case 64: return fp8::launch_tn<64>(L, stream);
    case 128: return fp8::launch_tn<128>(L, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace bsk
