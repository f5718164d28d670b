// kernels.h -- internal interface between the C-ABI layer (api.cu) and the
// kernel translation units.  Not installed; the public ABI is bsgemm.h.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace bsk {

// Launch with the library's attributes: programmatic stream serialization
// (the kernel may start while the previous kernel on the stream finishes; each
// kernel waits with griddepcontrol.wait before touching global memory another
// kernel may use) and, for cluster > 1, a 1-D cluster shape.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                          int cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

enum { kEpiStore = 0, kEpiSwiglu = 1, kEpiCombine = 2, kEpiRows = 3, kEpiSwigluQ4 = 4 };
// SWIGLU and SWIGLU_Q4 share the tile map (gate / up column blocks); Q4 then
// quantizes h in the epilogue instead of storing it.
constexpr bool epi_is_swiglu(int e) { return e == kEpiSwiglu || e == kEpiSwigluQ4; }

struct Fp4Params {
  const uint8_t* sfa;
  const uint8_t* sfb;
  int M, N, K;            // N: output columns
  float alpha;
  const float* col_scale; // [N] or null
  const void* bias;       // bf16 [N] or null
  void* out;
  int out_bf16;
  long long ldo;
  // grouped (E > 0)
  int E;
  const int* offsets;     // [E+1]
  const int* counts;      // [E]
  const int* token_of;
  const float* weight_of;
  float* out32;
  long long ld_out32;
  int* status;
  int n_chunk;            // grouped tile order: column blocks per chunk (0 = all)
  int part;               // grouped rows covered: 0 all, 1 experts > 128 rows, 2 the others (expert_part)
  int half_tail;          // dense, CTA pairs: split a short last wave into 256 x 128 half tiles
  uint8_t* out_sf;        // SWIGLU_Q4: scales of h (MMA layout for [M, N]); out holds its codes [M, N/2]
  unsigned long long wait_ns;  // bound of every pipeline wait (%globaltimer ns)
  const float* a_ts;      // two-level FP4: tensor scales of A / B (device fp32, or null = 1)
  const float* b_ts;
};

// Rows of expert e that one grouped launch covers.  part 0: all of them.  A
// grouped GEMM on CTA pairs is split in two launches so that small experts do
// not fill 256-row pair tiles with padding: part 1 (CTA pairs) takes the
// experts with more than 128 rows, part 2 (one CTA per 128-row tile) those
// with at most 128.  Whole experts move, so each expert's weights are still
// streamed by one launch only.
__device__ __forceinline__ void expert_part(const Fp4Params& p, int e, int& off, int& cnt) {
  off = p.offsets[e];
  cnt = p.counts[e];
  if (p.part == 0) return;
  const bool small = cnt <= 128;
  if ((p.part == 1 && small) || (p.part == 2 && !small)) cnt = 0;
}
struct Fp4Launch {
  CUtensorMap tmA, tmB, tmT, tmL;
  Fp4Params p;
  bool lora;
  int epilogue;
  int grid;
  int bk;                 // K elements per pipeline stage: 128 or 256 (tensor maps must match)
};

cudaError_t launch_fp4_gemm(const Fp4Launch& L, cudaStream_t stream);
int fp4_stages(bool lora, int bk);

// CTA-pair (cta_group::2) variant: K stages of 128, scales through TMA maps
// (uint32 view of the MMA scale layout, one row per 128-row block).
struct Fp4PairLaunch {
  Fp4Launch base;         // tmA/tmB built for 128-element stages; base.grid unused
  CUtensorMap tmSfa, tmSfb;
  CUtensorMap tmO;        // output boxes (dense STORE, SWIGLU); unused otherwise
  int grid;               // even: two CTAs per cluster
};
cudaError_t launch_fp4_pair_gemm(const Fp4PairLaunch& L, cudaStream_t stream);
int fp4_pair_stages(bool lora, int bk);

// FP4 decode shapes (M <= 32): swap-AB, stream-K over all SMs.
// Multi-weight launches: G <= kMaxProducts products Y_g = X W_g^T that share
// the token operand X, one weight tensor map per product.
constexpr int kMaxProducts = 8;
struct WeightMaps {
  CUtensorMap m[kMaxProducts];
};
// The weight-map kernel parameter: one map, or one per product.
template <bool kMulti>
struct WArg {
  using type = CUtensorMap;
};
template <>
struct WArg<true> {
  using type = WeightMaps;
};
// a[g] of a per-product parameter array, read with constant indices only (no
// local-memory copy of the parameter)
template <typename T>
__device__ __forceinline__ T pick(const T (&a)[kMaxProducts], int g) {
  T r = a[0];
#pragma unroll
  for (int i = 1; i < kMaxProducts; ++i)
    if (g == i) r = a[i];
  return r;
}

struct Fp4DecodeParams {
  const uint8_t* sfw;     // weight scales, MMA layout for [N, K]
  const uint8_t* sfx;     // token scales, MMA layout for [M, K] (block 0 holds every row)
  int M, N, K;
  float alpha;
  const float* col_scale; // [N] or null
  const void* bias;       // bf16 [N] or null
  const float* a_ts;      // two-level tensor scales (device, or null = 1)
  const float* b_ts;
  void* out;
  int out_bf16;
  long long ldo;
  float* work;            // stream-K partials [tiles][maxc][128][TN]
  int* counters;          // one arrival counter per tile (zero between calls)
  int maxc;
  int pre_b;              // weight stages loaded before waiting on the preceding kernel
  int* status;
  unsigned long long wait_ns;
  int G;                  // products sharing the tokens: 1 = one GEMM (sfw, out); > 1 = sfw_g, out_g
  const uint8_t* sfw_g[kMaxProducts];
  void* out_g[kMaxProducts];
};
struct Fp4DecodeLaunch {
  CUtensorMap tmW, tmX;
  WeightMaps tmW_g;       // G > 1: the weight map of every product (tmW unused)
  Fp4DecodeParams p;
  int tile_n;             // 16 or 32 token columns
  int grid;
};
cudaError_t launch_fp4_decode(const Fp4DecodeLaunch& L, cudaStream_t stream);
int fp4_decode_stages(int tile_n);

struct Fp8Params {
  const float* sfa;       // [K/128, M]
  const float* sfb;       // [ceil(N/128), K/128]
  int M, N, K;
  void* out;
  int out_bf16;
  long long ldo;
  float* work;            // stream-K: fp32 partials [tiles][maxc][128][TN]
  int* counters;          // stream-K: one arrival counter per tile (zero between calls)
  int stream_k;           // 1: the tiles' K blocks are shared out evenly over the grid
  int maxc;               // stream-K: most CTAs that share one tile
  int pre_b;              // weight stages loaded before waiting on the preceding kernel
  int rowwise;            // W8A8: sfa fp32 [M] per token, sfb fp32 [N] per channel; no per-block promotion
  int* status;
  unsigned long long wait_ns;  // bound of every pipeline wait (%globaltimer ns)
  int G;                  // products sharing the activation: 1 = one GEMM (sfb, out); > 1 = the
                          // multi-weight kernel (sfb_g, out_g; block scaling, M <= 32)
  const float* sfb_g[kMaxProducts];
  void* out_g[kMaxProducts];
};

struct Fp8Launch {
  CUtensorMap tmA, tmB;
  WeightMaps tmA_g;       // G > 1: the weight map of every product (tmA unused)
  Fp8Params p;
  int tile_n;             // MMA N (token columns per tile): 16, 32, 64 or 128
  int grid;
};

cudaError_t launch_fp8_gemm(const Fp8Launch& L, cudaStream_t stream);
int fp8_tile_n(long long M);
int fp8_stages(int tile_n);

// FP8 grouped over MoE experts: the tokens of a 128-row block of an expert
// segment are the MMA's M, kFp8GroupedBN weight rows its N.
constexpr int kFp8GroupedBN = 128;
struct Fp8GroupedParams {
  const float* sfa;       // [K/128, M]
  const float* sfb;       // [E * Nw / 128, K/128] (Nw = 2N for SWIGLU, else N)
  int M, N, K, E;         // N: output columns per row (SWIGLU: h columns)
  const int* offsets;     // [E+1]
  const int* counts;      // [E]
  const float* weight_of; // ROWS: [M]
  void* out;
  int out_bf16;
  long long ldo;
  int* status;
  unsigned long long wait_ns;  // bound of every pipeline wait (%globaltimer ns)
};
struct Fp8GroupedLaunch {
  CUtensorMap tmA;        // token codes [M, K], box 128 rows x 128 bytes
  CUtensorMap tmB;        // stacked weights [E * Nw, K], box kFp8GroupedBN / 2 rows x 128 bytes
  Fp8GroupedParams p;
  int epilogue;           // kEpiStore, kEpiSwiglu or kEpiRows
  int grid;
};
cudaError_t launch_fp8_grouped(const Fp8GroupedLaunch& L, cudaStream_t stream);
int fp8_grouped_stages();

// quantizers
cudaError_t launch_q4_quantize(const void* x, int x_bf16, long long M, long long K, long long ldx,
                               const int* gather, uint8_t* codes, uint8_t* sf, cudaStream_t stream,
                               const float* tensor_amax = nullptr, float* tensor_scale = nullptr);
cudaError_t launch_tensor_amax(const void* x, int x_bf16, long long M, long long K, long long ldx, float* amax,
                               cudaStream_t stream);
cudaError_t launch_q4_lowrank_fused(const void* x, long long M, long long K, long long ldx, const int* gather,
                                    const void* lora_a_t, uint8_t* codes, uint8_t* sf, void* lora_t,
                                    cudaStream_t stream);
cudaError_t launch_fp4_gather_rows(const uint8_t* codes_in, const uint8_t* sf_in, long long rows_in, long long K,
                                   const int* gather, long long rows_out, uint8_t* codes_out, uint8_t* sf_out,
                                   cudaStream_t stream);
cudaError_t launch_fp8_gather_rows(const uint8_t* codes_in, const float* scales_in, long long rows_in, long long K,
                                   const int* gather, long long rows_out, uint8_t* codes_out, float* scales_out,
                                   cudaStream_t stream);
cudaError_t launch_lowrank_t(const void* x, long long M, long long K, long long ldx, const int* gather,
                             const void* lora_a_t, void* lora_t, cudaStream_t stream);
cudaError_t launch_q8_quantize(const void* x, int x_bf16, long long M, long long K, long long ldx, int mode,
                               uint8_t* codes, float* scales, cudaStream_t stream);

// MoE
cudaError_t launch_moe_router(const float* logits, long long T, int E, int k, int* ids, float* w,
                              cudaStream_t stream);
cudaError_t launch_moe_dispatch(const int* topk_ids, const float* topk_w, long long T, int k, int E,
                                int* counts, int* offsets, int* pair_of_row, int* token_of, float* weight_of,
                                int* work, long long rows_bound, int* status, cudaStream_t stream);
cudaError_t launch_moe_finalize(float* out32, void* out_bf16, long long n, cudaStream_t stream);
cudaError_t launch_moe_combine(const float* rows, long long ld_rows, const int* pair_of_row, long long n_rows,
                               long long T, int k, long long H, int* row_of_pair, void* out, long long ldo,
                               cudaStream_t stream);

// Unique id of the CUDA context current on this thread (0 if none); keys the
// caches of device addresses of the library's __device__ variables.
unsigned long long current_context_id();

// Grouping whose histogram scratch is the library's static device array.
constexpr size_t kNoAllocDispatchScratchBytes = size_t(1) << 20;
cudaError_t launch_moe_dispatch_noalloc(const int* topk_ids, const float* topk_w, long long T, int k, int E,
                                        int* counts, int* offsets, int* pair_of_row, int* token_of,
                                        float* weight_of, long long rows_bound, int* status, cudaStream_t stream);

}  // namespace bsk
