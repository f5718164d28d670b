// moe.cu -- grouping of routed (token, slot) pairs by expert and the final
// fp32 -> bf16 cast of the combined MoE output.
//
// Grouping ("DeepGEMM teardown (FP8 GEMM)", section 5.3: pass group offsets,
// keep each expert's rows contiguous and movable in blocks) is a stable
// counting sort over the flattened pair index p = t*k + slot:
//   1. count:  one CTA per chunk of 1024 pairs -> histogram [chunk][E]
//   2. scan:   one CTA: per-expert running sums over chunks (stable bases),
//              counts, and 128-aligned segment offsets
//   3. place:  one CTA per chunk, each warp a 128-pair slice in order; ranks
//              among equal experts inside each 32-pair round come from
//              __match_any_sync and warp bases from a prefix over the warps,
//              so the result is identical to a sequential stable sort;
//              padding rows get pair/token -1 and weight 0
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace bsk {

constexpr int kChunk = 1024;
constexpr int kSegAlign = 128;

constexpr int kDispatchThreads = 256;  // 8 warps per chunk

__global__ void __launch_bounds__(kDispatchThreads) moe_count_kernel(const int* __restrict__ ids, long long P, int E,
                                                                     int* __restrict__ hist, int* status) {
  griddep_wait();  // inputs may come from the kernel just before on the stream
  griddep_launch_dependents();
  extern __shared__ int cnt[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const long long p0 = (long long)blockIdx.x * kChunk;
  for (int i = threadIdx.x; i < kChunk; i += blockDim.x) {
    const long long p = p0 + i;
    if (p >= P) break;
    const int e = ids[p];
    if (e < 0 || e >= E) {
      record_status(status, kStatusOffsets, 2);
      continue;
    }
    atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(long long)blockIdx.x * E + e] = cnt[e];
}

__global__ void __launch_bounds__(1024) moe_scan_kernel(int* __restrict__ hist, int nchunks, int E,
                                                        int* __restrict__ counts, int* __restrict__ offsets) {
  griddep_wait();  // inputs may come from the kernel just before on the stream
  griddep_launch_dependents();
  __shared__ int padded[1024];
  __shared__ int warp_sums[32];
  const int e = threadIdx.x;
  int total = 0;
  if (e < E) {
    // exclusive base of chunk c inside expert e; the counts of 16 chunks are
    // loaded together so their round trips overlap
    int c = 0;
    for (; c + 16 <= nchunks; c += 16) {
      int h[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) h[i] = hist[(long long)(c + i) * E + e];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        hist[(long long)(c + i) * E + e] = total;
        total += h[i];
      }
    }
    for (; c < nchunks; ++c) {
      const int h = hist[(long long)c * E + e];
      hist[(long long)c * E + e] = total;
      total += h;
    }
    counts[e] = total;
  }
  const int pad = (e < E) ? (total + kSegAlign - 1) / kSegAlign * kSegAlign : 0;
  // block-wide exclusive scan of the padded sizes
  const int lane = e & 31, warp = e >> 5;
  int incl = pad;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
    int wi = w;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, wi, d);
      if (lane >= d) wi += v;
    }
    warp_sums[lane] = wi - w;
  }
  __syncthreads();
  const int excl = warp_sums[warp] + incl - pad;
  padded[e] = excl;
  if (e < E) offsets[e] = excl;
  if (e == E - 1) offsets[E] = excl + pad;
  __syncthreads();
  if (e < E)
    for (int c = 0; c < nchunks; ++c) hist[(long long)c * E + e] += padded[e];
}

// Placement of one chunk by 8 warps: warp w owns pairs [128 w, 128 w + 128) of
// the chunk.  Its first position for expert e is the chunk's base plus the
// counts of warps 0 .. w-1 for e (a prefix over warps in shared memory); inside
// the warp, 32-pair rounds in order with __match_any_sync ranks.  The result
// equals a sequential stable sort.
__global__ void __launch_bounds__(kDispatchThreads) moe_place_kernel(
    const int* __restrict__ ids, const float* __restrict__ w, long long P, int k, int E, const int* __restrict__ base,
    const int* __restrict__ counts, const int* __restrict__ offsets, int* __restrict__ pair_of_row,
    int* __restrict__ token_of, float* __restrict__ weight_of, long long rows_bound) {
  griddep_wait();  // inputs may come from the kernel just before on the stream
  griddep_launch_dependents();
  extern __shared__ int pos[];  // [8][E]: per-warp counts, then per-warp running positions
  constexpr int kWarps = kDispatchThreads / 32;
  constexpr int kPerWarp = kChunk / kWarps;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int i = threadIdx.x; i < kWarps * E; i += blockDim.x) pos[i] = 0;
  __syncthreads();
  const long long p0 = (long long)blockIdx.x * kChunk + (long long)warp * kPerWarp;
  for (int i = lane; i < kPerWarp; i += 32) {
    const long long p = p0 + i;
    if (p < P) {
      const int e = ids[p];
      if (e >= 0 && e < E) atomicAdd(&pos[warp * E + e], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = base[(long long)blockIdx.x * E + e];
    for (int v = 0; v < kWarps; ++v) {
      const int c = pos[v * E + e];
      pos[v * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  int* my = pos + warp * E;
  for (int i = 0; i < kPerWarp; i += 32) {
    const long long p = p0 + i + lane;
    const bool live = p < P;
    int e = live ? ids[p] : -1;
    if (e >= E) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int leader = __ffs(peers) - 1;
    int slot = 0;
    if (e >= 0) slot = my[e] + rank;
    __syncwarp();
    if (e >= 0 && lane == leader) my[e] += __popc(peers);
    __syncwarp();
    if (e >= 0) {
      pair_of_row[slot] = (int)p;
      token_of[slot] = (int)(p / k);
      weight_of[slot] = w[p];
    }
  }
  // padding rows: a share of [0, rows_bound) per CTA
  const long long per = (rows_bound + gridDim.x - 1) / gridDim.x;
  const long long r0 = (long long)blockIdx.x * per;
  const long long r1 = min(rows_bound, r0 + per);
  for (long long r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
    bool pad_row = r >= offsets[E];
    if (!pad_row) {
      int lo = 0, hi = E - 1;  // largest e with offsets[e] <= r
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (offsets[mid] <= r) lo = mid; else hi = mid - 1;
      }
      pad_row = r >= (long long)offsets[lo] + counts[lo];
    }
    if (pad_row) {
      pair_of_row[r] = -1;
      token_of[r] = -1;
      weight_of[r] = 0.0f;
    }
  }
}

// out = bf16(out32), eight elements per thread: two 16-byte loads, one
// 16-byte store.  The zeroing of out32 is a separate pass: writing zeros back
// over the lines a thread has just read, in the same kernel, ran several
// times slower than the two streaming passes together on GB300.
__global__ void moe_cast_kernel(const float* __restrict__ out32, __nv_bfloat16* __restrict__ out, long long n) {
  griddep_wait();  // inputs may come from the kernel just before on the stream
  griddep_launch_dependents();
  const long long n8 = n / 8;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const float4 a = reinterpret_cast<const float4*>(out32)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(out32)[2 * i + 1];
    uint4 o;
    o.x = pack_bf16x2(a.x, a.y);
    o.y = pack_bf16x2(a.z, a.w);
    o.z = pack_bf16x2(b.x, b.y);
    o.w = pack_bf16x2(b.z, b.w);
    reinterpret_cast<uint4*>(out)[i] = o;
  }
  for (long long i = n8 * 8 + (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = __float2bfloat16_rn(out32[i]);
}

__global__ void moe_zero_kernel(float* __restrict__ out32, long long n) {
  griddep_wait();  // inputs may come from the kernel just before on the stream
  griddep_launch_dependents();
  const long long n4 = n / 4;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride)
    reinterpret_cast<float4*>(out32)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (long long i = n4 * 4 + (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) out32[i] = 0.0f;
}

// Top-k routing of each token from its fp32 router logits ("DeepGEMM for
// Hopper MoE", section 1: the gate scores the experts, the top k are chosen
// and weighted by a softmax of their scores).  One warp per token; lane l
// holds logits l, l + 32, ... (E <= 1024, so at most 32 per lane) and a mask
// of those not yet chosen.  Round j takes the warp's arg-max -- the larger
// logit, the lower expert id between equal ones -- so the experts come out in
// descending order exactly as a stable sort would give them; lane j keeps
// the j-th pick.  Weights: exp(l_j - l_0) / sum over the k picks, in fp32.
template <int NV>  // logits per lane: ceil(E / 32) rounded up to a power of two
__global__ void __launch_bounds__(256) moe_router_kernel(const float* __restrict__ logits, long long T, int E, int k,
                                                         int* __restrict__ ids, float* __restrict__ w) {
  griddep_wait();  // inputs may come from the kernel just before on the stream
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long t = (long long)blockIdx.x * 8 + threadIdx.x / 32;
  if (t >= T) return;
  const float* row = logits + t * E;
  float v[NV];
  uint32_t live = 0;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? __ldg(row + e) : 0.0f;
    live |= (e < E ? 1u : 0u) << i;
  }
  constexpr int kNone = 0x7fffffff;
  float my_v = 0.0f;
  int my_e = -1;
  for (int j = 0; j < k; ++j) {
    float bv = 0.0f;
    int be = kNone;
#pragma unroll
    for (int i = 0; i < NV; ++i)  // increasing expert id: strict > keeps the lower id of equal logits
      if (((live >> i) & 1u) && (be == kNone || v[i] > bv)) {
        bv = v[i];
        be = lane + 32 * i;
      }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, d);
      const int oe = __shfl_xor_sync(0xffffffffu, be, d);
      if (oe != kNone && (be == kNone || ov > bv || (ov == bv && oe < be))) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) live &= ~(1u << (be >> 5));
    if (lane == j) {
      my_v = bv;
      my_e = be;
    }
  }
  const float top = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = lane < k ? expf(my_v - top) : 0.0f;
  float sum = ex;
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, d);
  if (lane < k) {
    ids[t * k + lane] = my_e;
    w[t * k + lane] = __fdiv_rn(ex, sum);
  }
}

cudaError_t launch_moe_router(const float* logits, long long T, int E, int k, int* ids, float* w,
                              cudaStream_t stream) {
  const unsigned blocks = (unsigned)((T + 7) / 8 > 0 ? (T + 7) / 8 : 1);
  const int per_lane = (E + 31) / 32;
  if (per_lane <= 1) return launch_kernel(moe_router_kernel<1>, blocks, 256, 0, stream, 1, logits, T, E, k, ids, w);
  if (per_lane <= 2) return launch_kernel(moe_router_kernel<2>, blocks, 256, 0, stream, 1, logits, T, E, k, ids, w);
  if (per_lane <= 4) return launch_kernel(moe_router_kernel<4>, blocks, 256, 0, stream, 1, logits, T, E, k, ids, w);
  if (per_lane <= 8) return launch_kernel(moe_router_kernel<8>, blocks, 256, 0, stream, 1, logits, T, E, k, ids, w);
  if (per_lane <= 16) return launch_kernel(moe_router_kernel<16>, blocks, 256, 0, stream, 1, logits, T, E, k, ids, w);
  return launch_kernel(moe_router_kernel<32>, blocks, 256, 0, stream, 1, logits, T, E, k, ids, w);
}

long long moe_chunks(long long P) { return (P + kChunk - 1) / kChunk; }

cudaError_t launch_moe_dispatch(const int* topk_ids, const float* topk_w, long long T, int k, int E, int* counts,
                                int* offsets, int* pair_of_row, int* token_of, float* weight_of, int* work,
                                long long rows_bound, int* status, cudaStream_t stream) {
  const long long P = T * k;
  const long long nch = moe_chunks(P) > 0 ? moe_chunks(P) : 1;
  const size_t smem = (size_t)E * sizeof(int);
  const size_t smem_place = (size_t)(kDispatchThreads / 32) * E * sizeof(int);  // <= 32 KB for E <= 1024
  cudaError_t e = launch_kernel(moe_count_kernel, (unsigned)nch, kDispatchThreads, smem, stream, 1, topk_ids, P, E,
                                work, status);
  if (e != cudaSuccess) return e;
  e = launch_kernel(moe_scan_kernel, 1, 1024, 0, stream, 1, work, (int)nch, E, counts, offsets);
  if (e != cudaSuccess) return e;
  return launch_kernel(moe_place_kernel, (unsigned)nch, kDispatchThreads, smem_place, stream, 1, topk_ids, topk_w, P, k,
                       E, (const int*)work, (const int*)counts, (const int*)offsets, pair_of_row, token_of, weight_of,
                       rows_bound);
}

// row_of_pair = inverse of pair_of_row (-1 where no row holds the pair)
__global__ void moe_rows_init_kernel(int* __restrict__ row_of_pair, long long P) {
  griddep_wait();  // inputs may come from the kernel just before on the stream
  griddep_launch_dependents();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long p = (long long)blockIdx.x * blockDim.x + threadIdx.x; p < P; p += stride) row_of_pair[p] = -1;
}
__global__ void moe_rows_invert_kernel(const int* __restrict__ pair_of_row, long long n_rows,
                                       int* __restrict__ row_of_pair, long long P) {
  griddep_wait();  // inputs may come from the kernel just before on the stream
  griddep_launch_dependents();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long r = (long long)blockIdx.x * blockDim.x + threadIdx.x; r < n_rows; r += stride) {
    const int p = pair_of_row[r];
    if (p >= 0 && p < P) row_of_pair[p] = (int)r;
  }
}

// out[t, 8g .. 8g+8) = bf16(sum_j rows[row_of_pair[t*k + j], 8g .. 8g+8)), fp32
// sum in slot order.  One thread per (token, 8 columns); the slots are read in
// batches of 8 whose 16 loads are independent (that many 16-byte loads in
// flight per thread), then added in order.
constexpr int kCombineBatch = 8;
__global__ void __launch_bounds__(256) moe_combine_kernel(const float* __restrict__ rows, long long ld_rows,
                                                          const int* __restrict__ row_of_pair, long long T, int k,
                                                          long long G, __nv_bfloat16* __restrict__ out,
                                                          long long ldo) {
  griddep_wait();  // inputs may come from the kernel just before on the stream
  griddep_launch_dependents();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < T * G; i += stride) {
    const long long t = i / G, g = i % G;
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = 0.0f;
    for (int j0 = 0; j0 < k; j0 += kCombineBatch) {
      float4 lo[kCombineBatch], hi[kCombineBatch];
#pragma unroll
      for (int j = 0; j < kCombineBatch; ++j) {
        const int r = j0 + j < k ? row_of_pair[t * k + j0 + j] : -1;
        lo[j] = hi[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r >= 0) {
          const float4* src = reinterpret_cast<const float4*>(rows + (long long)r * ld_rows + g * 8);
          lo[j] = __ldg(src);
          hi[j] = __ldg(src + 1);
        }
      }
#pragma unroll
      for (int j = 0; j < kCombineBatch; ++j) {  // slot order; absent slots add +0
        acc[0] += lo[j].x; acc[1] += lo[j].y; acc[2] += lo[j].z; acc[3] += lo[j].w;
        acc[4] += hi[j].x; acc[5] += hi[j].y; acc[6] += hi[j].z; acc[7] += hi[j].w;
      }
    }
    *reinterpret_cast<uint4*>(out + t * ldo + g * 8) =
        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                   pack_bf16x2(acc[6], acc[7]));
  }
}

cudaError_t launch_moe_combine(const float* rows, long long ld_rows, const int* pair_of_row, long long n_rows,
                               long long T, int k, long long H, int* row_of_pair, void* out, long long ldo,
                               cudaStream_t stream) {
  auto grid = [](long long units) {
    long long b = (units + 255) / 256;
    return (unsigned)(b > 8192 ? 8192 : (b < 1 ? 1 : b));
  };
  const long long P = T * k;
  cudaError_t e = launch_kernel(moe_rows_init_kernel, grid(P), 256, 0, stream, 1, row_of_pair, P);
  if (e != cudaSuccess) return e;
  e = launch_kernel(moe_rows_invert_kernel, grid(n_rows), 256, 0, stream, 1, pair_of_row, n_rows, row_of_pair, P);
  if (e != cudaSuccess) return e;
  const long long G = H / 8;
  __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out);
  return launch_kernel(moe_combine_kernel, grid(T * G), 256, 0, stream, 1, rows, ld_rows, (const int*)row_of_pair, T,
                       k, G, o, ldo);
}

cudaError_t launch_moe_finalize(float* out32, void* out_bf16, long long n, cudaStream_t stream) {
  auto grid = [](long long units) {
    long long b = (units + 255) / 256;
    return (unsigned)(b > 4096 ? 4096 : (b < 1 ? 1 : b));
  };
  cudaError_t e = launch_kernel(moe_cast_kernel, grid(n / 8), 256, 0, stream, 1, (const float*)out32,
                                reinterpret_cast<__nv_bfloat16*>(out_bf16), n);
  if (e != cudaSuccess) return e;
  return launch_kernel(moe_zero_kernel, grid(n / 4), 256, 0, stream, 1, out32, n);
}

}  // namespace bsk

namespace bsk {

// ---------------------------------------------------------------------------
// Grouping with library-owned scratch, for callers that cannot allocate.
//
// The histogram / stable-base table of the grouping lives in this fixed
// device array instead of a caller-provided workspace.  Every GPU that loads
// the library keeps the array until the process exits.  All calls share it
// and it keeps whatever the last call left there; the count step overwrites
// every entry the later steps read, so nothing has to be cleared first.
// Calls whose kernels overlap on the GPU (two streams, or two threads) race
// on the array and must be serialised by the caller.
// ---------------------------------------------------------------------------
static __device__ __align__(256) int g_dispatch_scratch[kNoAllocDispatchScratchBytes / sizeof(int)];

namespace {
std::mutex g_scratch_mu;
struct ScratchAddr {
  unsigned long long ctx_id;  // context the address belongs to (0: not looked up)
  int* ptr;
};
ScratchAddr g_scratch[64] = {};
}  // namespace

// Device address of the array in the current context.  In host code the
// array's name is only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress once per context (a device's primary context, or any
// other context the caller makes current on it) and cached under the
// context's unique id; a call from a context other than the cached one looks
// the address up again.
cudaError_t dispatch_scratch_ptr(int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  unsigned long long ctx = current_context_id();
  if (ctx == 0 || g_scratch[dev].ctx_id != ctx) {
    int* p = nullptr;
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_dispatch_scratch);
    if (e != cudaSuccess) return e;
    g_scratch[dev] = ScratchAddr{current_context_id(), p};
  }
  *out = g_scratch[dev].ptr;
  return cudaSuccess;
}

cudaError_t launch_moe_dispatch_noalloc(const int* topk_ids, const float* topk_w, long long T, int k, int E,
                                        int* counts, int* offsets, int* pair_of_row, int* token_of,
                                        float* weight_of, long long rows_bound, int* status, cudaStream_t stream) {
  int* scratch = nullptr;
  cudaError_t e = dispatch_scratch_ptr(&scratch);
  if (e != cudaSuccess) return e;
  return launch_moe_dispatch(topk_ids, topk_w, T, k, E, counts, offsets, pair_of_row, token_of, weight_of, scratch,
                             rows_bound, status, stream);
}

}  // namespace bsk
