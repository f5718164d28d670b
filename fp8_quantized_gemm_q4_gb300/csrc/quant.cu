// quant.cu -- activation / weight quantizers for sm_103a.
//
// FP4: per group of 16 K elements s = e4m3(fl32(amax / 6)), code =
// e2m1(fl32(x / s)) ("Tencent AI Infra interview notes": E2M1 format table,
// per-group quantization, online activation quantization).  One lane owns one
// 16-element group; the quotients x / s are correctly rounded (one-correction
// form on packed fp32 pairs, or IEEE division), scales and codes are written
// at their places in the MMA layouts.  Codes use the hardware cvt with round
// to nearest even and saturation.
//
// FP8: s = fl32(amax / 448), code = e4m3(fl32(x / s)) per 1x128 token block or
// 128x128 weight block ("DeepGEMM teardown (FP8 GEMM)", sections 2.2 and 5.2).
//
// Low-rank left factor T = X A of L(X) = X A B ("Warp-specialised W4A4
// kernel", section 1) on the unquantized bf16 rows, fp32 accumulation on the
// warp-level tensor-core path, written as bf16 hi|lo pairs.
#include "kernels.h"
#include "ptx.cuh"

namespace bsk {

// quot_rn (correctly rounded group quotient) lives in ptx.cuh, shared with
// the GEMM epilogue that quantizes h.

__device__ __forceinline__ void load8(const void* x, int x_bf16, long long off, float (&v)[8]) {
  if (x_bf16) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(x) + off));
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else {
    const float4 a = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(x) + off));
    const float4 b = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(x) + off + 4));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

static int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

// 8 consecutive inputs as raw words: bf16 -> 4 words (pairs), fp32 -> 8 words.
template <bool kBf16>
struct Raw8 {
  uint32_t w[kBf16 ? 4 : 8];
};
template <bool kBf16>
__device__ __forceinline__ void load_raw8(const void* x, long long off, Raw8<kBf16>& r) {
  if constexpr (kBf16) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(x) + off));
    r.w[0] = u.x; r.w[1] = u.y; r.w[2] = u.z; r.w[3] = u.w;
  } else {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const float*>(x) + off));
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const float*>(x) + off + 4));
    r.w[0] = a.x; r.w[1] = a.y; r.w[2] = a.z; r.w[3] = a.w;
    r.w[4] = b.x; r.w[5] = b.y; r.w[6] = b.z; r.w[7] = b.w;
  }
}
template <bool kBf16>
__device__ __forceinline__ float raw8_at(const Raw8<kBf16>& r, int i) {
  if constexpr (kBf16)
    return __uint_as_float((i & 1) ? (r.w[i / 2] & 0xFFFF0000u) : (r.w[i / 2] << 16));
  else
    return __uint_as_float(r.w[i]);
}

// Two-level FP4 tensor scale 2^e: the smallest e with amax <= 6 * 448 * 2^e
// (0 for a zero tensor), decided with exact double comparisons.
// With 2688 = 21 * 2^7: amax <= 2688 * 2^e  <=>  amax * 2^-(e+7) <= 21, and the
// scaled value stays near 21, a normal fp32 number, so ldexpf is exact.
__device__ __forceinline__ int two_level_exp(float amax) {
  if (!(amax > 0.0f)) return 0;
  int e = ilogbf(amax) - 11;  // 2688 lies in [2^11, 2^12): at most a step or two off
  while (ldexpf(amax, -(e + 7)) > 21.0f) ++e;
  while (ldexpf(amax, -(e + 6)) <= 21.0f) --e;  // amax <= 2688 * 2^(e-1)
  return e;
}

// (s, RN(1/s)) of every e4m3 scale code, one table per CTA in shared memory
// (codes 0x7F / 0xFF are NaN and never produced by the saturating scale
// conversion; code 0 gives s = 0, whose groups are all zero codes).
__device__ __forceinline__ void fill_scale_table(float2* tab) {
  for (int c = threadIdx.x; c < 256; c += blockDim.x) {
    const float s = e4m3_to_f32((uint32_t)c);
    tab[c] = make_float2(s, __frcp_rn(s));
  }
}

// FP4 quantization of one 16-element group held as eight fp32 pairs (exact
// values of the input): scale code e4m3(RN(amax / 6)), codes E2M1 RNE of
// RN(x / s) (all +0 when s == 0), element i in nibble i of the result.
//
// The quotient is quot_rn's one-correction form on pairs (packed fp32x2
// multiply-add): p = RN(x r), rem = x - p s (exact), q = RN(p + r rem).  The
// remainder is rounded downward: its value is exact either way, but an exact
// zero then comes out as -0, so that q keeps the sign of a -0 input (the
// zero remainder of +0 gives -0 * r + 0 = +0), with no copysign per element.
// kBf16Amax: amax is a bf16 value and RN(amax / 6) is quot_rn's form (checked
// exhaustively on the GPU); otherwise IEEE division.
__device__ __forceinline__ float fmax3(float a, float b, float c) {  // three-input max (sm_100 family)
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

template <bool kBf16Amax>
__device__ __forceinline__ uint64_t q4_group16_x2(const float2 (&x)[8], const float2* tab, uint32_t& sc) {
  // |x| max as a tree of three-input maxes (depth 3, not a chain of 8)
  float m[6];
#pragma unroll
  for (int i = 0; i < 5; ++i) {
    const int a = 3 * i, b = 3 * i + 1, c = 3 * i + 2;
    m[i] = fmax3(fabsf(a % 2 ? x[a / 2].y : x[a / 2].x), fabsf(b % 2 ? x[b / 2].y : x[b / 2].x),
                 fabsf(c % 2 ? x[c / 2].y : x[c / 2].x));
  }
  m[5] = fabsf(x[7].y);
  const float amax = fmax3(fmax3(m[0], m[1], m[2]), m[3], fmaxf(m[4], m[5]));
  float a6;
  if constexpr (kBf16Amax) {
    const float r6 = __frcp_rn(6.0f);
    const float p = amax * r6;
    a6 = fmaf(fmaf(-p, 6.0f, amax), r6, p);  // amax >= 0: no sign of zero to keep
  } else {
    a6 = __fdiv_rn(amax, 6.0f);
  }
  sc = f32_to_e4m3(a6);
  const float2 sr = tab[sc];
  const float2 r2 = make_float2(sr.y, sr.y), ns2 = make_float2(-sr.x, -sr.x);
  float q[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 p = __fmul2_rn(x[i], r2);
    const float2 rem = __ffma2_rd(p, ns2, x[i]);
    const float2 qq = __ffma2_rn(rem, r2, p);
    q[2 * i] = qq.x;
    q[2 * i + 1] = qq.y;
  }
  const float(&lo)[8] = *reinterpret_cast<const float(*)[8]>(&q[0]);
  const float(&hi)[8] = *reinterpret_cast<const float(*)[8]>(&q[8]);
  if (sr.x == 0.0f) return 0ull;  // zero group: all codes +0
  return (uint64_t)f32x8_to_e2m1x8(lo) | ((uint64_t)f32x8_to_e2m1x8(hi) << 32);
}

// One lane per 16-element group: a warp covers 512 consecutive elements of a
// row per segment and kQ4Seg segments per work item, every load of the item
// issued before any arithmetic (4 KB in flight per warp for bf16 input).
// Codes: 8 bytes per lane (a warp's 256 bytes contiguous); scales: one byte
// per lane at its place in the MMA scale layout.  Rows in [M, Mpad) (the
// 128-row padding of the scale tensor) get zero scales, no codes.
//
// kScaled: two-level FP4, the input divided by the tensor scale 2^e first
// (exact: a multiply by an fp32 power of two, or ldexpf where 2^-e is not an
// fp32 normal), e derived from *tensor_amax; CTA 0 stores 2^e.
constexpr int kQ4Seg = 4;
template <bool kBf16, bool kScaled>
__global__ void __launch_bounds__(256, kBf16 ? 3 : 2) q4_quantize_kernel(const void* __restrict__ x, long long M, long long Mpad,
                                                          long long K, long long ldx,
                                                          const int* __restrict__ gather,
                                                          uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                          const float* __restrict__ tensor_amax,
                                                          float* __restrict__ tensor_scale) {
  __shared__ float2 tab[256];
  __shared__ int e2_s;
  fill_scale_table(tab);  // before the dependency wait: touches no global memory
  griddep_wait();         // inputs may come from the kernel just before on the stream
  griddep_launch_dependents();
  if (kScaled && threadIdx.x == 0) {
    e2_s = two_level_exp(__ldg(tensor_amax));  // once per CTA
    if (blockIdx.x == 0) *tensor_scale = ldexpf(1.0f, e2_s);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  int e2 = 0;
  float down = 1.0f;
  bool fast = true;
  if constexpr (kScaled) {
    e2 = e2_s;
    fast = e2 >= -126 && e2 <= 126;
    down = fast ? ldexpf(1.0f, -e2) : 1.0f;
  }
  constexpr int NW = kBf16 ? 8 : 16;  // 32-bit words per group
  const long long nseg = (K + 512 * kQ4Seg - 1) / (512 * kQ4Seg);
  const long long total = Mpad * nseg;
  const long long kchunks = K / 64;
  for (long long w = (long long)blockIdx.x * 8 + threadIdx.x / 32; w < total; w += (long long)gridDim.x * 8) {
    const long long row = w / nseg, seg = w % nseg;
    long long src = row < M ? row : -1;
    if (src >= 0 && gather) src = gather[row];
    uint32_t raw[kQ4Seg][NW];
#pragma unroll
    for (int u = 0; u < kQ4Seg; ++u) {
      const long long k0 = ((seg * kQ4Seg + u) * 32 + lane) * 16;
#pragma unroll
      for (int i = 0; i < NW; ++i) raw[u][i] = 0u;
      if (k0 < K && src >= 0) {
        const uint4* p = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(x) +
                                                        (src * ldx + k0) * (kBf16 ? 2 : 4));
#pragma unroll
        for (int j = 0; j < NW / 4; ++j) {
          const uint4 v = __ldg(p + j);
          raw[u][4 * j] = v.x;
          raw[u][4 * j + 1] = v.y;
          raw[u][4 * j + 2] = v.z;
          raw[u][4 * j + 3] = v.w;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kQ4Seg; ++u) {
      const long long g = (seg * kQ4Seg + u) * 32 + lane;  // group index within the row
      const long long k0 = g * 16;
      if (k0 >= K) continue;
      float2 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if constexpr (kBf16)
          v[i] = make_float2(__uint_as_float(raw[u][i] << 16), __uint_as_float(raw[u][i] & 0xFFFF0000u));
        else
          v[i] = make_float2(__uint_as_float(raw[u][2 * i]), __uint_as_float(raw[u][2 * i + 1]));
        if constexpr (kScaled) {
          if (fast) v[i] = __fmul2_rn(v[i], make_float2(down, down));
          else v[i] = make_float2(ldexpf(v[i].x, -e2), ldexpf(v[i].y, -e2));
        }
      }
      uint32_t sc;
      const uint64_t cw = q4_group16_x2<kBf16>(v, tab, sc);
      if (row < M) *reinterpret_cast<uint2*>(codes + row * (K / 2) + k0 / 2) = make_uint2((uint32_t)cw, (uint32_t)(cw >> 32));
      const long long off = ((row / 128) * kchunks + g / 4) * 512 + (row % 32) * 16 + ((row % 128) / 32) * 4 + g % 4;
      sf[off] = (uint8_t)sc;  // padding rows: an all-zero group, scale code 0
    }
  }
}

// T[m, j] = sum_k x[src(m), k] * At[j, k] for j < 32, on mma.sync m16n8k16
// (bf16 x bf16 -> fp32).  A CTA owns 16 rows; its 8 warps interleave the K
// steps and reduce through shared memory.  Output bf16 [M, 64]: hi | lo.
__global__ void __launch_bounds__(256) lowrank_t_kernel(const __nv_bfloat16* __restrict__ x, long long M,
                                                        long long K, long long ldx,
                                                        const int* __restrict__ gather,
                                                        const __nv_bfloat16* __restrict__ at,
                                                        __nv_bfloat16* __restrict__ t_out) {
  griddep_wait();  // inputs may come from the kernel just before on the stream
  griddep_launch_dependents();
  __shared__ float red[8][16][33];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane / 4, tq = lane % 4;
  const long long r0 = (long long)blockIdx.x * 16;
  long long src_lo = r0 + g < M ? r0 + g : -1, src_hi = r0 + g + 8 < M ? r0 + g + 8 : -1;
  if (gather) {
    if (src_lo >= 0) src_lo = gather[src_lo];
    if (src_hi >= 0) src_hi = gather[src_hi];
  }
  const uint32_t* xlo = src_lo >= 0 ? reinterpret_cast<const uint32_t*>(x + src_lo * ldx) : nullptr;
  const uint32_t* xhi = src_hi >= 0 ? reinterpret_cast<const uint32_t*>(x + src_hi * ldx) : nullptr;
  float d[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) d[i][j] = 0.0f;
  for (long long k = (long long)warp * 16; k < K; k += 8 * 16) {
    const long long c0 = (k + 2 * tq) / 2, c1 = (k + 2 * tq + 8) / 2;  // uint32 (bf16 pair) index
    const uint32_t a0 = xlo ? __ldg(xlo + c0) : 0u, a1 = xhi ? __ldg(xhi + c0) : 0u;
    const uint32_t a2 = xlo ? __ldg(xlo + c1) : 0u, a3 = xhi ? __ldg(xhi + c1) : 0u;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const uint32_t* brow = reinterpret_cast<const uint32_t*>(at + (long long)(nt * 8 + g) * K);
      const uint32_t b0 = __ldg(brow + c0), b1 = __ldg(brow + c1);
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
          "{%0, %1, %2, %3};"
          : "+f"(d[nt][0]), "+f"(d[nt][1]), "+f"(d[nt][2]), "+f"(d[nt][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
  }
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    red[warp][g][nt * 8 + 2 * tq] = d[nt][0];
    red[warp][g][nt * 8 + 2 * tq + 1] = d[nt][1];
    red[warp][g + 8][nt * 8 + 2 * tq] = d[nt][2];
    red[warp][g + 8][nt * 8 + 2 * tq + 1] = d[nt][3];
  }
  __syncthreads();
  for (int o = threadIdx.x; o < 16 * 32; o += 256) {
    const int rr = o / 32, j = o % 32;
    const long long row = r0 + rr;
    if (row >= M) continue;
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += red[w][rr][j];
    const __nv_bfloat16 hi = __float2bfloat16_rn(s);
    const __nv_bfloat16 lo = __float2bfloat16_rn(s - __bfloat162float(hi));
    t_out[row * 64 + j] = hi;
    t_out[row * 64 + 32 + j] = lo;
  }
}

// FP8 1x128 per token.  Each lane owns 8 consecutive elements (one 16-byte
// bf16 load, two for fp32), 16 lanes a 128-element block, so a warp covers
// two blocks of one row per 256-element unit; a warp takes kQ8Unroll units of
// a row and issues all their loads before any arithmetic (4 KB of bf16 in
// flight per warp).  The block amax is a 4-step shuffle over the 16 lanes;
// s = fl32(amax / 448) and every code's quotient x / s use IEEE division.
// (The one-correction quotient of the FP4 quantizers is exact for their e4m3
// scales, checked exhaustively; for arbitrary fp32 scales it is not always
// correctly rounded, which the quotient sweep over 512 scales shows.)
constexpr int kQ8Unroll = 8;
template <bool kBf16>
__global__ void __launch_bounds__(256) q8_token_kernel(const void* __restrict__ x, long long M, long long K,
                                                       long long ldx, uint8_t* __restrict__ codes,
                                                       float* __restrict__ scales) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long units = (K + 255) / 256;
  const long long ngrp = (units + kQ8Unroll - 1) / kQ8Unroll;
  const long long total = M * ngrp;
  for (long long w = (long long)blockIdx.x * 8 + threadIdx.x / 32; w < total; w += (long long)gridDim.x * 8) {
    const long long row = w / ngrp, g = w % ngrp;
    Raw8<kBf16> raw[kQ8Unroll];
#pragma unroll
    for (int u = 0; u < kQ8Unroll; ++u) {
      const long long k0 = (g * kQ8Unroll + u) * 256 + lane * 8;
#pragma unroll
      for (int i = 0; i < (kBf16 ? 4 : 8); ++i) raw[u].w[i] = 0u;
      if (k0 < K) load_raw8<kBf16>(x, row * ldx + k0, raw[u]);
    }
#pragma unroll
    for (int u = 0; u < kQ8Unroll; ++u) {
      const long long k0 = (g * kQ8Unroll + u) * 256 + lane * 8;
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(raw8_at<kBf16>(raw[u], i)));
#pragma unroll
      for (int d = 1; d < 16; d <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
      if (k0 >= K) continue;  // after the shuffles: the whole warp takes part in them
      const float s = __fdiv_rn(amax, 448.0f);
      uint32_t c[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float q[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] = s == 0.0f ? 0.0f : __fdiv_rn(raw8_at<kBf16>(raw[u], 4 * h + i), s);
        c[h] = f32x2_to_e4m3x2(q[0], q[1]) | (f32x2_to_e4m3x2(q[2], q[3]) << 16);
      }
      *reinterpret_cast<uint2*>(codes + row * K + k0) = make_uint2(c[0], c[1]);
      if ((lane & 15) == 0) scales[(k0 / 128) * M + row] = s;
    }
  }
}

// FP8 with one scale per row over all of K (W8A8: per-token activations,
// per-channel weights held as [N, K] rows).  One CTA per row: a first pass
// takes the row's amax (16-byte loads, block reduction), s = fl32(amax / 448);
// a second pass (the row is now in L2) writes the codes, IEEE division.
template <bool kBf16>
__global__ void __launch_bounds__(256) q8_row_kernel(const void* __restrict__ x, long long M, long long K,
                                                     long long ldx, uint8_t* __restrict__ codes,
                                                     float* __restrict__ scales) {
  griddep_wait();  // inputs may come from the kernel just before on the stream
  griddep_launch_dependents();
  __shared__ float wmax[8];
  for (long long row = blockIdx.x; row < M; row += gridDim.x) {
    const long long base = row * ldx;
    float m = 0.0f;
    for (long long k = (long long)threadIdx.x * 8; k < K; k += 256 * 8) {
      Raw8<kBf16> r;
      load_raw8<kBf16>(x, base + k, r);
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(raw8_at<kBf16>(r, i)));
    }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x / 32] = m;
    __syncthreads();
    float amax = wmax[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) amax = fmaxf(amax, wmax[w]);
    __syncthreads();  // wmax is reused by the next row
    const float s = __fdiv_rn(amax, 448.0f);
    if (threadIdx.x == 0) scales[row] = s;
    for (long long k = (long long)threadIdx.x * 8; k < K; k += 256 * 8) {
      Raw8<kBf16> r;
      load_raw8<kBf16>(x, base + k, r);
      uint32_t c[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float q[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] = s == 0.0f ? 0.0f : __fdiv_rn(raw8_at<kBf16>(r, 4 * h + i), s);
        c[h] = f32x2_to_e4m3x2(q[0], q[1]) | (f32x2_to_e4m3x2(q[2], q[3]) << 16);
      }
      *reinterpret_cast<uint2*>(codes + row * K + k) = make_uint2(c[0], c[1]);
    }
  }
}

// FP8 128x128 blocks: one CTA (256 threads) per block.
__global__ void __launch_bounds__(256) q8_block_kernel(const void* __restrict__ x, int x_bf16, long long M,
                                                       long long K, long long ldx, uint8_t* __restrict__ codes,
                                                       float* __restrict__ scales) {
  __shared__ float wmax[8];
  griddep_wait();
  griddep_launch_dependents();
  const long long rb = blockIdx.x / (K / 128), kb = blockIdx.x % (K / 128);
  const int tid = threadIdx.x;
  // thread -> (row r = tid / 2 .. in 2 passes of 64 rows? keep it simple: 64 elements each)
  const int r_local = tid / 2, c_local = (tid % 2) * 64;
  const long long row = rb * 128 + r_local;
  float v[64];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 64; i += 8) {
    float t8[8];
    if (row < M) {
      load8(x, x_bf16, row * ldx + kb * 128 + c_local + i, t8);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) t8[j] = 0.0f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[i + j] = t8[j];
      amax = fmaxf(amax, fabsf(t8[j]));
    }
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
  if ((tid & 31) == 0) wmax[tid / 32] = amax;
  __syncthreads();
  amax = wmax[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, wmax[i]);
  const float s = __fdiv_rn(amax, 448.0f);
  if (tid == 0) scales[rb * (K / 128) + kb] = s;
  if (row < M) {
#pragma unroll
    for (int i = 0; i < 64; i += 16) {
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float q0 = (s == 0.0f) ? 0.0f : __fdiv_rn(v[i + 4 * j], s);
        const float q1 = (s == 0.0f) ? 0.0f : __fdiv_rn(v[i + 4 * j + 1], s);
        const float q2 = (s == 0.0f) ? 0.0f : __fdiv_rn(v[i + 4 * j + 2], s);
        const float q3 = (s == 0.0f) ? 0.0f : __fdiv_rn(v[i + 4 * j + 3], s);
        w[j] = f32x2_to_e4m3x2(q0, q1) | (f32x2_to_e4m3x2(q2, q3) << 16);
      }
      *reinterpret_cast<uint4*>(codes + row * K + kb * 128 + c_local + i) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// max |x| over an [M, K] tensor into *amax: a one-thread kernel zeroes it,
// then every CTA reduces its grid-stride share and merges with an integer
// atomicMax (non-negative floats order like their bit patterns).
__global__ void tensor_amax_init_kernel(float* amax) {
  griddep_wait();
  griddep_launch_dependents();
  *amax = 0.0f;
}
template <bool kBf16>
__global__ void __launch_bounds__(256) tensor_amax_kernel(const void* __restrict__ x, long long M, long long K,
                                                          long long ldx, float* __restrict__ amax) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float wmax[8];
  const long long per_row = K / 8, total = M * per_row;
  float m = 0.0f;
  for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < total; v += (long long)gridDim.x * blockDim.x) {
    Raw8<kBf16> r;
    load_raw8<kBf16>(x, (v / per_row) * ldx + (v % per_row) * 8, r);
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(raw8_at<kBf16>(r, i)));
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x / 32] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < 8; ++w) m = fmaxf(m, wmax[w]);
    atomicMax(reinterpret_cast<unsigned int*>(amax), __float_as_uint(m));
  }
}

cudaError_t launch_tensor_amax(const void* x, int x_bf16, long long M, long long K, long long ldx, float* amax,
                               cudaStream_t stream) {
  cudaError_t e = launch_kernel(tensor_amax_init_kernel, 1, 1, 0, stream, 1, amax);
  if (e != cudaSuccess) return e;
  long long blocks = (M * (K / 8) + 255) / 256;
  const long long cap = (long long)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (x_bf16) return launch_kernel(tensor_amax_kernel<true>, (unsigned)blocks, 256, 0, stream, 1, x, M, K, ldx, amax);
  return launch_kernel(tensor_amax_kernel<false>, (unsigned)blocks, 256, 0, stream, 1, x, M, K, ldx, amax);
}

cudaError_t launch_q4_quantize(const void* x, int x_bf16, long long M, long long K, long long ldx,
                               const int* gather, uint8_t* codes, uint8_t* sf, cudaStream_t stream,
                               const float* tensor_amax, float* tensor_scale) {
  const long long Mpad = (M + 127) / 128 * 128;
  const long long warps = Mpad * ((K + 512 * kQ4Seg - 1) / (512 * kQ4Seg));
  long long blocks = (warps + 7) / 8;
  const long long cap = (long long)sm_count() * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (tensor_amax) {
    if (x_bf16)
      return launch_kernel(q4_quantize_kernel<true, true>, (unsigned)blocks, 256, 0, stream, 1, x, M, Mpad, K, ldx,
                           gather, codes, sf, tensor_amax, tensor_scale);
    return launch_kernel(q4_quantize_kernel<false, true>, (unsigned)blocks, 256, 0, stream, 1, x, M, Mpad, K, ldx,
                         gather, codes, sf, tensor_amax, tensor_scale);
  }
  if (x_bf16)
    return launch_kernel(q4_quantize_kernel<true, false>, (unsigned)blocks, 256, 0, stream, 1, x, M, Mpad, K, ldx,
                         gather, codes, sf, tensor_amax, tensor_scale);
  return launch_kernel(q4_quantize_kernel<false, false>, (unsigned)blocks, 256, 0, stream, 1, x, M, Mpad, K, ldx,
                       gather, codes, sf, tensor_amax, tensor_scale);
}

cudaError_t launch_lowrank_t(const void* x, long long M, long long K, long long ldx, const int* gather,
                             const void* lora_a_t, void* lora_t, cudaStream_t stream) {
  const long long blocks = (M + 15) / 16;
  return launch_kernel(lowrank_t_kernel, (unsigned)blocks, 256, 0, stream, 1,
                       reinterpret_cast<const __nv_bfloat16*>(x), M, K, ldx, gather,
                       reinterpret_cast<const __nv_bfloat16*>(lora_a_t), reinterpret_cast<__nv_bfloat16*>(lora_t));
}

cudaError_t launch_q8_quantize(const void* x, int x_bf16, long long M, long long K, long long ldx, int mode,
                               uint8_t* codes, float* scales, cudaStream_t stream) {
  if (mode == 1) {
    const long long warps = M * (((K + 255) / 256 + kQ8Unroll - 1) / kQ8Unroll);
    long long blocks = (warps + 7) / 8;
    const long long cap = (long long)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (x_bf16) return launch_kernel(q8_token_kernel<true>, (unsigned)blocks, 256, 0, stream, 1, x, M, K, ldx, codes, scales);
    return launch_kernel(q8_token_kernel<false>, (unsigned)blocks, 256, 0, stream, 1, x, M, K, ldx, codes, scales);
  }
  if (mode == 3) {  // one scale per row over all of K
    long long blocks = M < (long long)sm_count() * 8 ? M : (long long)sm_count() * 8;
    if (blocks < 1) blocks = 1;
    if (x_bf16) return launch_kernel(q8_row_kernel<true>, (unsigned)blocks, 256, 0, stream, 1, x, M, K, ldx, codes, scales);
    return launch_kernel(q8_row_kernel<false>, (unsigned)blocks, 256, 0, stream, 1, x, M, K, ldx, codes, scales);
  }
  // one CTA per 128 x 128 block, numbered kb + (K / 128) * rb
  return launch_kernel(q8_block_kernel, (unsigned)((K / 128) * ((M + 127) / 128)), 256, 0, stream, 1, x, x_bf16, M,
                       K, ldx, codes, scales);
}

}  // namespace bsk

namespace bsk {

// ---------------------------------------------------------------------------
// Fused FP4 quantization + low-rank left factor for bf16 rows.
//
// One CTA of 8 R threads owns R = 16 rows and streams them through shared
// memory in K chunks of 256 (2-stage cp.async ring: 8 KB of X + 16 KB of A^T
// per stage, ~50 KB per CTA so four CTAs share an SM and all 512 CTAs of an
// 8192-row matrix are resident at once: each does half the work of a 32-row
// CTA, with as many warps per SM).  Each 16-byte chunk j of row r is stored at
// chunk position j ^ (r % 8).  Per stage:
//   - quantization: thread t owns row t % R and the 32-element piece t / R of
//     the chunk (two groups: half of a 32-bit word of the MMA scale layout,
//     written as 16 bits, and 16 bytes of codes); the row swizzle keeps the
//     lanes of a warp on distinct banks;
//   - low rank: warp w multiplies rows 16 (w % RG) .. +16 by A over K quarter
//     w / RG of the chunk with ldmatrix + mma.sync m16n8k16 (bf16 -> fp32); the
//     four K quarters are summed through shared memory at the end and T is
//     written as bf16 hi | lo.
// X is read from HBM once for both results.
// ---------------------------------------------------------------------------
namespace fq {
constexpr int R = 16;          // rows per CTA
constexpr int NT = 8 * R;      // threads: eight 32-element pieces of a K chunk per row
constexpr int KC = 256;        // K per stage
constexpr int S = 2;           // stages
constexpr int XB = R * KC * 2;       // 8 KB
constexpr int AB = 32 * KC * 2;      // 16 KB
constexpr int RG = R / 16;           // 16-row groups of the low-rank MMA; each has 4 K-quarter warps
static_assert(NT / 32 == 4 * RG, "four K quarters per row group");
constexpr int STAGE = XB + AB;
constexpr int RED = 4 * R * 32 * 4;  // [4 K quarters][R rows][32] fp32, in the stage buffers after the loop
constexpr int TAB = 256 * 8;         // (s, 1/s) of every e4m3 scale code
constexpr int SMEM = S * STAGE + TAB;
static_assert(RED <= S * STAGE, "reduction buffer reuses the stages");
}  // namespace fq

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* g, bool valid) {
  const int n = valid ? 16 : 0;  // src-size 0 -> zero fill
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(saddr), "l"(g), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t saddr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(saddr));
}

// byte offset of 16-byte chunk `chunk` of row `row` in a [rows][KC] bf16 tile
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * (fq::KC * 2) + ((chunk ^ (row & 7)) * 16));
}

__global__ void __launch_bounds__(fq::NT, 4) q4_lowrank_fused_kernel(
    const __nv_bfloat16* __restrict__ x, long long M, long long Mpad, long long K, long long ldx,
    const int* __restrict__ gather, const __nv_bfloat16* __restrict__ at, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ sf, __nv_bfloat16* __restrict__ t_out) {
  extern __shared__ __align__(128) uint8_t fsm[];
  float2* tab = reinterpret_cast<float2*>(fsm + fq::S * fq::STAGE);
  fill_scale_table(tab);  // read after the first stage barrier below
  griddep_wait();         // inputs may come from the kernel just before on the stream
  griddep_launch_dependents();
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const long long r0 = (long long)blockIdx.x * fq::R;
  const int nchunks = (int)(K / fq::KC);
  const uint32_t sbase = smem_u32(fsm);

  // loader: X chunk = R rows x 32 chunks of 16 B (4 copies per thread);
  // A^T chunk = 32 rows x 32 chunks (1024 / NT copies per thread)
  constexpr int XC = fq::R * 32 / fq::NT, AC = 32 * 32 / fq::NT;
  long long my_src[XC];
#pragma unroll
  for (int i = 0; i < XC; ++i) {
    const long long row = r0 + (tid + i * fq::NT) / 32;
    my_src[i] = row >= M ? -1 : (gather ? (long long)gather[row] : row);
  }
  auto load_stage = [&](int c, int st) {
    const uint32_t xs = sbase + st * fq::STAGE, as = xs + fq::XB;
    const long long k0 = (long long)c * fq::KC;
#pragma unroll
    for (int i = 0; i < XC; ++i) {
      const int idx = tid + i * fq::NT, r = idx / 32, ch = idx % 32;
      const long long sr = my_src[i];
      const __nv_bfloat16* g = x + (sr >= 0 ? sr * ldx + k0 + ch * 8 : 0);
      cp_async16(xs + swz(r, ch), g, sr >= 0);
    }
#pragma unroll
    for (int i = 0; i < AC; ++i) {
      const int idx = tid + i * fq::NT, r = idx / 32, ch = idx % 32;
      cp_async16(as + swz(r, ch), at + (long long)r * K + k0 + ch * 8, true);
    }
  };

  // quantization role: row qrow, 32-element piece qp (chunks 4 qp .. 4 qp + 3)
  const int qrow = tid % fq::R, qp = tid / fq::R;
  const long long grow = r0 + qrow;
  // low-rank role of this warp: rows 16 rg .. +16, K quarter kq (64 elements)
  const int rg = warp % fq::RG, kq = warp / fq::RG;
  float d[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) d[i][j] = 0.0f;

  for (int st = 0; st < fq::S - 1; ++st) {
    if (st < nchunks) load_stage(st, st);
    cp_async_commit();
  }
  for (int c = 0; c < nchunks; ++c) {
    const int st = c % fq::S;
    if (c + fq::S - 1 < nchunks) load_stage(c + fq::S - 1, (c + fq::S - 1) % fq::S);
    cp_async_commit();
    cp_async_wait<fq::S - 1>();
    __syncthreads();
    const uint32_t xs = sbase + st * fq::STAGE, as = xs + fq::XB;

    // ---- quantize 32 elements (2 groups) of row qrow
    {
      uint32_t raw[16];
      const uint8_t* xg = fsm + st * fq::STAGE;  // generic view of this stage's X tile
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 u = *reinterpret_cast<const uint4*>(xg + swz(qrow, qp * 4 + j));
        raw[4 * j] = u.x;
        raw[4 * j + 1] = u.y;
        raw[4 * j + 2] = u.z;
        raw[4 * j + 3] = u.w;
      }
      uint32_t sfh = 0;
      uint32_t cw[4];
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        float2 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          v[i] = make_float2(__uint_as_float(raw[8 * g + i] << 16), __uint_as_float(raw[8 * g + i] & 0xFFFF0000u));
        uint32_t sc;
        const uint64_t c2 = q4_group16_x2<true>(v, tab, sc);
        sfh |= sc << (8 * g);
        cw[2 * g] = (uint32_t)c2;
        cw[2 * g + 1] = (uint32_t)(c2 >> 32);
      }
      // two scale bytes = half of the 64-element chunk's scale word
      const long long kp = (long long)c * fq::KC + qp * 32;  // first element of the piece
      if (grow < Mpad) {
        const long long off = ((grow / 128) * (K / 64) + kp / 64) * 512 + (grow % 32) * 16 + ((grow % 128) / 32) * 4 +
                              ((kp / 32) & 1) * 2;
        *reinterpret_cast<uint16_t*>(sf + off) = (grow < M) ? (uint16_t)sfh : (uint16_t)0;
      }
      if (grow < M)
        *reinterpret_cast<uint4*>(codes + grow * (K / 2) + kp / 2) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
    }

    // ---- low rank: rows 16 rg .. +16, K quarter kq of the chunk (4 k-steps)
    {
      const int arow = rg * 16 + (lane % 16);
      const int ahalf = lane / 16;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const int kchunk = kq * 8 + ks * 2;  // 16-byte chunk of this k-step's first 8 elements
        uint32_t a0, a1, a2, a3;
        ldsm_x4(xs + swz(arow, kchunk + ahalf), a0, a1, a2, a3);
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          const int brow = np * 16 + (lane % 8) + ((lane / 16) * 8);
          const int bhalf = (lane / 8) % 2;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(as + swz(brow, kchunk + bhalf), b0, b1, b2, b3);
          asm volatile(
              "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
              "{%0, %1, %2, %3};"
              : "+f"(d[2 * np][0]), "+f"(d[2 * np][1]), "+f"(d[2 * np][2]), "+f"(d[2 * np][3])
              : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
          asm volatile(
              "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
              "{%0, %1, %2, %3};"
              : "+f"(d[2 * np + 1][0]), "+f"(d[2 * np + 1][1]), "+f"(d[2 * np + 1][2]), "+f"(d[2 * np + 1][3])
              : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b2), "r"(b3));
        }
      }
    }
    __syncthreads();  // stage st may be refilled next iteration
  }
  cp_async_wait<0>();

  // ---- reduce the four K quarters and write T as bf16 hi | lo (the last
  // loop iteration ended with a barrier and no copy is in flight, so the
  // stage buffers are free)
  float* red = reinterpret_cast<float*>(fsm);  // [4][32][32]
  {
    const int g = lane / 4, tq = lane % 4;
    float* rb = red + (kq * fq::R + rg * 16) * 32;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      rb[g * 32 + nt * 8 + 2 * tq] = d[nt][0];
      rb[g * 32 + nt * 8 + 2 * tq + 1] = d[nt][1];
      rb[(g + 8) * 32 + nt * 8 + 2 * tq] = d[nt][2];
      rb[(g + 8) * 32 + nt * 8 + 2 * tq + 1] = d[nt][3];
    }
  }
  __syncthreads();
  for (int o = tid; o < fq::R * 32; o += fq::NT) {
    const int r = o / 32, j = o % 32;
    const long long row = r0 + r;
    if (row >= M) continue;
    float t = 0.0f;
#pragma unroll
    for (int w = 0; w < 4; ++w) t += red[(w * fq::R + r) * 32 + j];
    const __nv_bfloat16 hi = __float2bfloat16_rn(t);
    const __nv_bfloat16 lo = __float2bfloat16_rn(t - __bfloat162float(hi));
    t_out[row * 64 + j] = hi;
    t_out[row * 64 + 32 + j] = lo;
  }
}

cudaError_t launch_q4_lowrank_fused(const void* x, long long M, long long K, long long ldx, const int* gather,
                                    const void* lora_a_t, uint8_t* codes, uint8_t* sf, void* lora_t,
                                    cudaStream_t stream) {
  const long long Mpad = (M + 127) / 128 * 128;
  const long long blocks = Mpad / fq::R;  // covers the scale padding rows too
  cudaError_t e = cudaFuncSetAttribute(q4_lowrank_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       fq::SMEM);
  if (e != cudaSuccess) return e;
  return launch_kernel(q4_lowrank_fused_kernel, (unsigned)blocks, fq::NT, (size_t)fq::SMEM, stream, 1,
                       reinterpret_cast<const __nv_bfloat16*>(x), M, Mpad, K, ldx, gather,
                       reinterpret_cast<const __nv_bfloat16*>(lora_a_t), codes, sf,
                       reinterpret_cast<__nv_bfloat16*>(lora_t));
}

}  // namespace bsk

namespace bsk {

// Gather rows of an already quantized FP4 matrix: out row i = in row
// gather[i] (negative: zero row), codes copied as 16-byte vectors, each
// 64-element chunk's scale word moved from the source row's place in the MMA
// scale layout to the destination row's.  Equal, bit for bit, to quantizing
// the gathered bf16 rows (quantization is row-local), at a fraction of the
// traffic when rows repeat (MoE: each token feeds k experts).
// One CTA per 128-row block of the output.  Codes: each warp copies 16 rows,
// a lane's 16-byte vectors of a row issued together.  Scales: the block's
// 512-byte word groups (one per 64-element chunk) are written whole — lane l
// of a chunk's warp stores the 16 bytes holding rows l, l + 32, l + 64 and
// l + 96 — so every store is a full coalesced line, and the four source
// words come from the (cache-resident) input scale rows.
constexpr int kGatherVec = 8;  // 16-byte code vectors in flight per lane and pass
__global__ void __launch_bounds__(256) fp4_gather_rows_kernel(const uint8_t* __restrict__ codes_in,
                                                              const uint8_t* __restrict__ sf_in, long long rows_in,
                                                              long long K, const int* __restrict__ gather,
                                                              long long rows_out, long long rows_out_pad,
                                                              uint8_t* __restrict__ codes_out,
                                                              uint8_t* __restrict__ sf_out) {
  griddep_wait();  // inputs may come from the kernel just before on the stream
  griddep_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long kv = K / 32;  // 16-byte vectors per row of codes
  const long long kc = K / 64;  // scale words per row
  for (long long blk = blockIdx.x; blk * 128 < rows_out_pad; blk += gridDim.x) {
    const long long r0 = blk * 128;
    // codes: warp w copies rows r0 + 16 w .. + 16 (their sources read up front)
    long long my_src = -1;
    if (lane < 16 && r0 + warp * 16 + lane < rows_out) {
      my_src = gather[r0 + warp * 16 + lane];
      if (my_src >= rows_in) my_src = -1;
    }
    const long long left = rows_out - (r0 + warp * 16);
    const int nrows = left < 16 ? (left > 0 ? (int)left : 0) : 16;
    // two rows per pass: both rows' loads are in flight before either is stored
    for (int i = 0; i < nrows; i += 2) {
      const bool two = i + 1 < nrows;
      const long long row = r0 + warp * 16 + i;
      const long long src0 = __shfl_sync(0xffffffffu, my_src, i);
      const long long src1 = __shfl_sync(0xffffffffu, my_src, two ? i + 1 : i);
      const uint4* sp0 = reinterpret_cast<const uint4*>(codes_in + (src0 >= 0 ? src0 : 0) * (K / 2));
      const uint4* sp1 = reinterpret_cast<const uint4*>(codes_in + (src1 >= 0 ? src1 : 0) * (K / 2));
      uint4* dp0 = reinterpret_cast<uint4*>(codes_out + row * (K / 2));
      uint4* dp1 = dp0 + kv;
      for (long long v0 = 0; v0 < kv; v0 += 32 * kGatherVec) {
        uint4 buf[2][kGatherVec];
#pragma unroll
        for (int u = 0; u < kGatherVec; ++u) {
          const long long v = v0 + u * 32 + lane;
          buf[0][u] = (src0 >= 0 && v < kv) ? __ldg(sp0 + v) : make_uint4(0, 0, 0, 0);
          buf[1][u] = (two && src1 >= 0 && v < kv) ? __ldg(sp1 + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kGatherVec; ++u) {
          const long long v = v0 + u * 32 + lane;
          if (v < kv) {
            __stcs(dp0 + v, buf[0][u]);  // streaming: keep the source rows in L2
            if (two) __stcs(dp1 + v, buf[1][u]);
          }
        }
      }
    }
    // scales: lane l serves rows r0 + l + 32 q (q = 0..3) of every chunk
    long long soff[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const long long row = r0 + lane + 32 * q;
      long long src = row < rows_out ? (long long)gather[row] : -1;
      if (src >= rows_in) src = -1;
      soff[q] = src < 0 ? -1 : (src / 128) * kc * 512 + (src % 32) * 16 + ((src % 128) / 32) * 4;
    }
    for (long long c = warp; c < kc; c += 8) {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        w[q] = soff[q] >= 0 ? __ldg(reinterpret_cast<const uint32_t*>(sf_in + soff[q] + c * 512)) : 0u;
      __stcs(reinterpret_cast<uint4*>(sf_out + (blk * kc + c) * 512 + lane * 16), make_uint4(w[0], w[1], w[2], w[3]));
    }
  }
}

cudaError_t launch_fp4_gather_rows(const uint8_t* codes_in, const uint8_t* sf_in, long long rows_in, long long K,
                                   const int* gather, long long rows_out, uint8_t* codes_out, uint8_t* sf_out,
                                   cudaStream_t stream) {
  const long long pad = (rows_out + 127) / 128 * 128;
  long long blocks = pad / 128;
  const long long cap = (long long)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_kernel(fp4_gather_rows_kernel, (unsigned)blocks, 256, 0, stream, 1, codes_in, sf_in, rows_in, K, gather,
                       rows_out, pad, codes_out, sf_out);
}

// Rows of an FP8 matrix written by q8_quantize in 1x128 token mode, gathered:
// output row i = input row gather[i] (negative or out of range: a zero row
// with zero scales).  The scales are K-block major ([K/128, rows]), so for
// each K block the 128 scales of an output row block are one coalesced
// 512-byte store.  Used to group MoE activations by expert after quantizing
// each token once ("DeepGEMM teardown", section 5.3).
__global__ void __launch_bounds__(256) fp8_gather_rows_kernel(const uint8_t* __restrict__ codes_in,
                                                              const float* __restrict__ scales_in,
                                                              long long rows_in, long long K,
                                                              const int* __restrict__ gather, long long rows_out,
                                                              uint8_t* __restrict__ codes_out,
                                                              float* __restrict__ scales_out) {
  griddep_wait();  // inputs may come from the kernel just before on the stream
  griddep_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long kv = K / 16;   // 16-byte vectors per row of codes
  const long long nkb = K / 128;
  for (long long blk = blockIdx.x; blk * 128 < rows_out; blk += gridDim.x) {
    const long long r0 = blk * 128;
    // codes: warp w copies rows r0 + 16 w .. + 16 (their sources read up front)
    long long my_src = -1;
    if (lane < 16 && r0 + warp * 16 + lane < rows_out) {
      my_src = gather[r0 + warp * 16 + lane];
      if (my_src >= rows_in) my_src = -1;
    }
    const long long left = rows_out - (r0 + warp * 16);
    const int nrows = left < 16 ? (left > 0 ? (int)left : 0) : 16;
    // two rows per pass: both rows' loads are in flight before either is stored
    for (int i = 0; i < nrows; i += 2) {
      const bool two = i + 1 < nrows;
      const long long row = r0 + warp * 16 + i;
      const long long src0 = __shfl_sync(0xffffffffu, my_src, i);
      const long long src1 = __shfl_sync(0xffffffffu, my_src, two ? i + 1 : i);
      const uint4* sp0 = reinterpret_cast<const uint4*>(codes_in + (src0 >= 0 ? src0 : 0) * K);
      const uint4* sp1 = reinterpret_cast<const uint4*>(codes_in + (src1 >= 0 ? src1 : 0) * K);
      uint4* dp0 = reinterpret_cast<uint4*>(codes_out + row * K);
      uint4* dp1 = dp0 + kv;
      for (long long v0 = 0; v0 < kv; v0 += 32 * kGatherVec) {
        uint4 buf[2][kGatherVec];
#pragma unroll
        for (int u = 0; u < kGatherVec; ++u) {
          const long long v = v0 + u * 32 + lane;
          buf[0][u] = (src0 >= 0 && v < kv) ? __ldg(sp0 + v) : make_uint4(0, 0, 0, 0);
          buf[1][u] = (two && src1 >= 0 && v < kv) ? __ldg(sp1 + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kGatherVec; ++u) {
          const long long v = v0 + u * 32 + lane;
          if (v < kv) {
            dp0[v] = buf[0][u];
            if (two) dp1[v] = buf[1][u];
          }
        }
      }
    }
    // scales: thread j serves row r0 + (j % 128) of every other K block
    const long long row = r0 + (tid & 127);
    long long src = row < rows_out ? (long long)gather[row] : -1;
    if (src >= rows_in) src = -1;
    if (row < rows_out) {
      for (long long kb = tid >> 7; kb < nkb; kb += 2)
        scales_out[kb * rows_out + row] = src >= 0 ? __ldg(scales_in + kb * rows_in + src) : 0.0f;
    }
  }
}

cudaError_t launch_fp8_gather_rows(const uint8_t* codes_in, const float* scales_in, long long rows_in, long long K,
                                   const int* gather, long long rows_out, uint8_t* codes_out, float* scales_out,
                                   cudaStream_t stream) {
  long long blocks = (rows_out + 127) / 128;
  const long long cap = (long long)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_kernel(fp8_gather_rows_kernel, (unsigned)blocks, 256, 0, stream, 1, codes_in, scales_in, rows_in, K,
                       gather, rows_out, codes_out, scales_out);
}

}  // namespace bsk
