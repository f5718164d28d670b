// api.cu -- the C ABI declared in include/bsgemm.h: host-side validation,
// TMA tensor-map encoding, the sticky device status word, and launches.
// Nothing here allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "bsgemm.h"
#include "kernels.h"

static_assert(BS_MOE_DISPATCH_NOALLOC_MAX_BYTES == bsk::kNoAllocDispatchScratchBytes,
              "header limit and static scratch size must agree");

namespace bsk {

// Unique id of the CUDA context current on the calling thread, 0 if none.
// Device addresses of the library's __device__ variables belong to a context
// (a non-primary context, or the primary context re-created after
// cudaDeviceReset, has its own), so address caches are keyed on this id, which
// the driver never reuses within a process.  The driver calls are reached
// through the runtime's entry-point query (no libcuda link).
unsigned long long current_context_id() {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id + 1;  // never 0 for a live context
}

}  // namespace bsk

namespace {

thread_local char g_err[512] = "";

bs_status fail(bs_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
bs_status fail(bs_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return s;
}

bs_status cuda_fail(cudaError_t e, const char* what) {
  return fail(BS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device status word: one per context, its address looked up once per
// context (see bsk::current_context_id).
__device__ int g_device_status;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct DeviceInfo {
  unsigned long long ctx_id;  // context the address below belongs to (0: not looked up)
  int* status;
  int sms;
};
DeviceInfo g_info[kMaxDevices] = {};

bool device_info(int** status, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  unsigned long long ctx = bsk::current_context_id();
  if (ctx == 0 || g_info[dev].ctx_id != ctx) {
    // first call in this context (or a context other than the cached one):
    // the lookup also makes the runtime's primary context current if none is
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return false;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    ctx = bsk::current_context_id();
    g_info[dev] = DeviceInfo{ctx, static_cast<int*>(p), n};
  }
  if (status) *status = g_info[dev].status;
  if (sms) *sms = g_info[dev].sms;
  return true;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D tiled map over a row-major [rows, inner] matrix.
bs_status make_map(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, uint64_t inner,
                   uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(BS_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  if (rows == 0) rows = 1;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  (void)esize;
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(BS_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return BS_OK;
}

}  // namespace

extern "C" {

size_t bs_sf_bytes(int64_t rows, int64_t K) {
  if (rows < 0 || K < 0) return 0;
  return (size_t)((rows + 127) / 128 * 128) * (size_t)(K / 16);
}

int64_t bs_sf_offset(int64_t row, int64_t group, int64_t K) {
  const int64_t kchunks = K / 64;
  return ((row / 128) * kchunks + group / 4) * 512 + (row % 32) * 16 + ((row % 128) / 32) * 4 + group % 4;
}

const char* bs_status_string(bs_status s) {
  switch (s) {
    case BS_OK: return "ok";
    case BS_ERR_INVALID: return "invalid argument";
    case BS_ERR_ALIGN: return "misaligned pointer, leading dimension or size";
    case BS_ERR_UNSUPPORTED: return "unsupported combination";
    case BS_ERR_CUDA: return "CUDA error";
    case BS_ERR_TIMEOUT: return "device pipeline wait timed out";
    case BS_ERR_OFFSETS: return "inconsistent expert offsets or ids";
  }
  return "unknown status";
}

const char* bs_last_error(void) { return g_err; }

bs_status bs_get_device_status(int* detail) {
  int* p = nullptr;
  if (!device_info(&p, nullptr)) return fail(BS_ERR_CUDA, "no current device");
  int v = 0;
  cudaError_t e = cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading device status");
  if (detail) *detail = v;
  return static_cast<bs_status>(v & 0xFF);
}

bs_status bs_clear_device_status(void) {
  int* p = nullptr;
  if (!device_info(&p, nullptr)) return fail(BS_ERR_CUDA, "no current device");
  int zero = 0;
  cudaError_t e = cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "clearing device status");
  return BS_OK;
}

bs_status q4_quantize(const void* x, bs_dtype dt, int64_t M, int64_t K, int64_t ldx, const int32_t* gather,
                      uint8_t* codes, uint8_t* sf, const void* lora_a_t, int r, void* lora_t,
                      bs_stream_t stream) {
  if (M < 0 || K <= 0) return fail(BS_ERR_INVALID, "q4_quantize: M=%lld K=%lld", (long long)M, (long long)K);
  if (dt != BS_DTYPE_F32 && dt != BS_DTYPE_BF16) return fail(BS_ERR_INVALID, "q4_quantize: dtype %d", (int)dt);
  if (K % 64) return fail(BS_ERR_ALIGN, "q4_quantize: K=%lld not a multiple of 64", (long long)K);
  if (M == 0) return BS_OK;
  if (!x || !codes || !sf) return fail(BS_ERR_INVALID, "q4_quantize: null pointer");
  if (ldx < K || ldx % 8 || !aligned16(x) || !aligned16(codes) || !aligned16(sf))
    return fail(BS_ERR_ALIGN, "q4_quantize: x/codes/sf must be 16-byte aligned and ldx %% 8 == 0, ldx >= K");
  const bool want_lora = lora_a_t || lora_t || r;
  if (want_lora) {
    if (!lora_a_t || !lora_t || r != 32) return fail(BS_ERR_INVALID, "q4_quantize: low-rank needs A^T, T and r == 32");
    if (dt != BS_DTYPE_BF16) return fail(BS_ERR_UNSUPPORTED, "q4_quantize: low-rank branch needs bf16 input");
    if (!aligned16(lora_a_t) || !aligned16(lora_t)) return fail(BS_ERR_ALIGN, "q4_quantize: low-rank buffers misaligned");
  }
  if (!device_info(nullptr, nullptr)) return fail(BS_ERR_CUDA, "no current device");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (want_lora && K % 256 == 0) {
    // one pass over X for codes, scales and T
    cudaError_t e = bsk::launch_q4_lowrank_fused(x, M, K, ldx, gather, lora_a_t, codes, sf, lora_t, s);
    if (e != cudaSuccess) return cuda_fail(e, "fused quantize + low-rank launch");
    return BS_OK;
  }
  cudaError_t e = bsk::launch_q4_quantize(x, dt == BS_DTYPE_BF16, M, K, ldx, gather, codes, sf, s);
  if (e != cudaSuccess) return cuda_fail(e, "q4_quantize launch");
  if (want_lora) {
    e = bsk::launch_lowrank_t(x, M, K, ldx, gather, lora_a_t, lora_t, s);
    if (e != cudaSuccess) return cuda_fail(e, "low-rank launch");
  }
  return BS_OK;
}

bs_status bs_tensor_amax(const void* x, bs_dtype dt, int64_t M, int64_t K, int64_t ldx, float* amax,
                         bs_stream_t stream) {
  if (M < 0 || K <= 0) return fail(BS_ERR_INVALID, "tensor_amax: M=%lld K=%lld", (long long)M, (long long)K);
  if (dt != BS_DTYPE_F32 && dt != BS_DTYPE_BF16) return fail(BS_ERR_INVALID, "tensor_amax: dtype %d", (int)dt);
  if (K % 8) return fail(BS_ERR_ALIGN, "tensor_amax: K=%lld not a multiple of 8", (long long)K);
  if (!amax || (M > 0 && !x)) return fail(BS_ERR_INVALID, "tensor_amax: null pointer");
  if ((M > 0 && (!aligned16(x) || ldx < K || ldx % 8)) || (reinterpret_cast<uintptr_t>(amax) & 3))
    return fail(BS_ERR_ALIGN, "tensor_amax: x 16-byte aligned with ldx %% 8 == 0 and ldx >= K, amax 4-byte aligned");
  if (!device_info(nullptr, nullptr)) return fail(BS_ERR_CUDA, "no current device");
  cudaError_t e = bsk::launch_tensor_amax(x, dt == BS_DTYPE_BF16, M, K, ldx, amax, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "tensor_amax launch");
  return BS_OK;
}

bs_status q4_quantize_two_level(const void* x, bs_dtype dt, int64_t M, int64_t K, int64_t ldx, const float* amax,
                                uint8_t* codes, uint8_t* sf, float* tensor_scale, bs_stream_t stream) {
  if (M < 0 || K <= 0) return fail(BS_ERR_INVALID, "q4_quantize_two_level: M=%lld K=%lld", (long long)M, (long long)K);
  if (dt != BS_DTYPE_F32 && dt != BS_DTYPE_BF16)
    return fail(BS_ERR_INVALID, "q4_quantize_two_level: dtype %d", (int)dt);
  if (K % 64) return fail(BS_ERR_ALIGN, "q4_quantize_two_level: K=%lld not a multiple of 64", (long long)K);
  if (!amax || !tensor_scale) return fail(BS_ERR_INVALID, "q4_quantize_two_level: null amax / tensor_scale");
  if ((reinterpret_cast<uintptr_t>(amax) | reinterpret_cast<uintptr_t>(tensor_scale)) & 3)
    return fail(BS_ERR_ALIGN, "q4_quantize_two_level: amax / tensor_scale must be 4-byte aligned");
  if (M == 0) return BS_OK;
  if (!x || !codes || !sf) return fail(BS_ERR_INVALID, "q4_quantize_two_level: null pointer");
  if (ldx < K || ldx % 8 || !aligned16(x) || !aligned16(codes) || !aligned16(sf))
    return fail(BS_ERR_ALIGN, "q4_quantize_two_level: x/codes/sf must be 16-byte aligned and ldx %% 8 == 0, ldx >= K");
  if (!device_info(nullptr, nullptr)) return fail(BS_ERR_CUDA, "no current device");
  cudaError_t e = bsk::launch_q4_quantize(x, dt == BS_DTYPE_BF16, M, K, ldx, nullptr, codes, sf,
                                          reinterpret_cast<cudaStream_t>(stream), amax, tensor_scale);
  if (e != cudaSuccess) return cuda_fail(e, "q4_quantize_two_level launch");
  return BS_OK;
}

bs_status bs_fp4_gather_rows(const uint8_t* codes_in, const uint8_t* sf_in, int64_t rows_in, int64_t K,
                             const int32_t* gather, int64_t rows_out, uint8_t* codes_out, uint8_t* sf_out,
                             bs_stream_t stream) {
  if (rows_in < 0 || rows_out < 0 || K <= 0) return fail(BS_ERR_INVALID, "gather_rows: bad sizes");
  if (K % 64) return fail(BS_ERR_ALIGN, "gather_rows: K=%lld not a multiple of 64", (long long)K);
  if (rows_out == 0) return BS_OK;
  if (!gather || !codes_out || !sf_out || (rows_in > 0 && (!codes_in || !sf_in)))
    return fail(BS_ERR_INVALID, "gather_rows: null pointer");
  if (!aligned16(codes_out) || !aligned16(sf_out) || (codes_in && !aligned16(codes_in)) || (sf_in && !aligned16(sf_in)))
    return fail(BS_ERR_ALIGN, "gather_rows: buffers must be 16-byte aligned");
  if (!device_info(nullptr, nullptr)) return fail(BS_ERR_CUDA, "no current device");
  cudaError_t e = bsk::launch_fp4_gather_rows(codes_in, sf_in, rows_in, K, gather, rows_out, codes_out, sf_out,
                                              reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gather_rows launch");
  return BS_OK;
}

bs_status bs_fp8_gather_rows(const uint8_t* codes_in, const float* scales_in, int64_t rows_in, int64_t K,
                             const int32_t* gather, int64_t rows_out, uint8_t* codes_out, float* scales_out,
                             bs_stream_t stream) {
  if (rows_in < 0 || rows_out < 0 || K <= 0) return fail(BS_ERR_INVALID, "fp8_gather_rows: bad sizes");
  if (K % 128) return fail(BS_ERR_ALIGN, "fp8_gather_rows: K=%lld not a multiple of 128", (long long)K);
  if (rows_out == 0) return BS_OK;
  if (!gather || !codes_out || !scales_out || (rows_in > 0 && (!codes_in || !scales_in)))
    return fail(BS_ERR_INVALID, "fp8_gather_rows: null pointer");
  if (!aligned16(codes_out) || (codes_in && !aligned16(codes_in)) ||
      ((reinterpret_cast<uintptr_t>(scales_out) | reinterpret_cast<uintptr_t>(scales_in)) & 3))
    return fail(BS_ERR_ALIGN, "fp8_gather_rows: codes must be 16-byte and scales 4-byte aligned");
  if (!device_info(nullptr, nullptr)) return fail(BS_ERR_CUDA, "no current device");
  cudaError_t e = bsk::launch_fp8_gather_rows(codes_in, scales_in, rows_in, K, gather, rows_out, codes_out,
                                              scales_out, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fp8_gather_rows launch");
  return BS_OK;
}

bs_status q8_quantize(const void* x, bs_dtype dt, int64_t M, int64_t K, int64_t ldx, int mode, uint8_t* codes,
                      float* scales, bs_stream_t stream) {
  if (M < 0 || K <= 0) return fail(BS_ERR_INVALID, "q8_quantize: M=%lld K=%lld", (long long)M, (long long)K);
  if (dt != BS_DTYPE_F32 && dt != BS_DTYPE_BF16) return fail(BS_ERR_INVALID, "q8_quantize: dtype %d", (int)dt);
  if (mode != BS_Q8_TOKEN_1x128 && mode != BS_Q8_BLOCK_128x128 && mode != BS_Q8_ROW)
    return fail(BS_ERR_INVALID, "q8_quantize: mode %d", mode);
  if (K % 128) return fail(BS_ERR_ALIGN, "q8_quantize: K=%lld not a multiple of 128", (long long)K);
  if (M == 0) return BS_OK;
  if (!x || !codes || !scales) return fail(BS_ERR_INVALID, "q8_quantize: null pointer");
  if (ldx < K || ldx % 8 || !aligned16(x) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(scales) & 3))
    return fail(BS_ERR_ALIGN, "q8_quantize: misaligned input/output or ldx");
  if (!device_info(nullptr, nullptr)) return fail(BS_ERR_CUDA, "no current device");
  cudaError_t e = bsk::launch_q8_quantize(x, dt == BS_DTYPE_BF16, M, K, ldx, mode, codes, scales,
                                          reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "q8_quantize launch");
  return BS_OK;
}

// Range checks of the per-call kernel choices (0 = default everywhere).
static bs_status check_choices(const bs_gemm_args* a) {
  if (a->fp4_kernel < 0 || a->fp4_kernel > 2) return fail(BS_ERR_INVALID, "fp4_kernel=%d (0, 1 or 2)", a->fp4_kernel);
  if (a->fp4_stage_k != 0 && a->fp4_stage_k != 128 && a->fp4_stage_k != 256)
    return fail(BS_ERR_INVALID, "fp4_stage_k=%d (0, 128 or 256)", a->fp4_stage_k);
  if (a->fp4_small_experts < 0 || a->fp4_small_experts > 2)
    return fail(BS_ERR_INVALID, "fp4_small_experts=%d (0, 1 or 2)", a->fp4_small_experts);
  if (a->fp4_half_tail < 0 || a->fp4_half_tail > 2)
    return fail(BS_ERR_INVALID, "fp4_half_tail=%d (0, 1 or 2)", a->fp4_half_tail);
  if (a->fp8_stream_k < 0 || a->fp8_stream_k > 2)
    return fail(BS_ERR_INVALID, "fp8_stream_k=%d (0, 1 or 2)", a->fp8_stream_k);
  if (a->weights_ready < 0 || a->weights_ready > 1) return fail(BS_ERR_INVALID, "weights_ready=%d (0 or 1)", a->weights_ready);
  if (a->fp8_scaling < 0 || a->fp8_scaling > 2) return fail(BS_ERR_INVALID, "fp8_scaling=%d (0, 1 or 2)", a->fp8_scaling);
  if (a->fp4_decode < 0 || a->fp4_decode > 2) return fail(BS_ERR_INVALID, "fp4_decode=%d (0, 1 or 2)", a->fp4_decode);
  if (a->wait_timeout_us < 0) return fail(BS_ERR_INVALID, "wait_timeout_us < 0");
  return BS_OK;
}

static bs_status check_common(const bs_gemm_args* a, bool grouped) {
  if (!a) return fail(BS_ERR_INVALID, "null args");
  if (a->M < 0 || a->N <= 0 || a->K <= 0) return fail(BS_ERR_INVALID, "bad sizes M=%lld N=%lld K=%lld",
                                                    (long long)a->M, (long long)a->N, (long long)a->K);
  if (a->M > (1LL << 30) || a->N > (1LL << 30) || a->K > (1LL << 30)) return fail(BS_ERR_INVALID, "sizes too large");
  if (a->N % 128) return fail(BS_ERR_ALIGN, "N=%lld not a multiple of 128", (long long)a->N);
  bs_status st = check_choices(a);
  if (st != BS_OK) return st;
  if (a->M == 0) return BS_OK;  // nothing to compute; operands may be empty (null)
  if (!a->a || !a->b || !a->sfa || !a->sfb) return fail(BS_ERR_INVALID, "null operand");
  if (!aligned16(a->a) || !aligned16(a->b) || !aligned16(a->sfa) || !aligned16(a->sfb))
    return fail(BS_ERR_ALIGN, "operands must be 16-byte aligned");
  if (!grouped || a->out) {
    if (!a->out) return fail(BS_ERR_INVALID, "null out");
    if (a->out_dtype != BS_DTYPE_F32 && a->out_dtype != BS_DTYPE_BF16) return fail(BS_ERR_INVALID, "out dtype");
    if (!aligned16(a->out) || a->ldo % 8 || a->ldo < a->N) return fail(BS_ERR_ALIGN, "out must be 16-byte aligned, ldo %% 8 == 0, ldo >= N");
  }
  if (a->num_sms < 0) return fail(BS_ERR_INVALID, "num_sms < 0");
  if (a->n_chunk_blocks < 0) return fail(BS_ERR_INVALID, "n_chunk_blocks < 0");
  return BS_OK;
}

// Pipeline-wait bound of the kernels launched for `a` (nanoseconds).
constexpr unsigned long long kDefaultWaitNs = 4000000000ull;  // 4 s
static unsigned long long wait_ns(const bs_gemm_args* a) {
  return a->wait_timeout_us > 0 ? (unsigned long long)a->wait_timeout_us * 1000ull : kDefaultWaitNs;
}

// FP4 stage depth: 256 K elements (128-byte rows, 128B swizzle) measured
// faster than 128 (64-byte rows) on GB300 even though the finer ring holds
// more stages.
static int fp4_bk(const bs_gemm_args* a) { return a->fp4_stage_k == 128 ? 128 : 256; }

static bs_status fp4_maps(bsk::Fp4Launch& L, const bs_gemm_args* a, int64_t b_rows, int bk) {
  const uint64_t kb = (uint64_t)a->K / 2;
  L.bk = bk;
  const uint32_t box = (uint32_t)L.bk / 2;
  const CUtensorMapSwizzle sw = L.bk == 256 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  bs_status st = make_map(&L.tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a->a, kb, (uint64_t)a->M, kb, box, 128, sw);
  if (st != BS_OK) return st;
  st = make_map(&L.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a->b, kb, (uint64_t)b_rows, kb, box, 128, sw);
  if (st != BS_OK) return st;
  if (a->lora_t) {
    st = make_map(&L.tmT, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a->lora_t, 64, (uint64_t)a->M, 128, 32, 128,
                  CU_TENSOR_MAP_SWIZZLE_64B);
    if (st != BS_OK) return st;
    st = make_map(&L.tmL, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a->lora_b_t, 32, (uint64_t)a->N, 64, 32, 128,
                  CU_TENSOR_MAP_SWIZZLE_64B);
    if (st != BS_OK) return st;
  } else {
    memset(&L.tmT, 0, sizeof L.tmT);
    memset(&L.tmL, 0, sizeof L.tmL);
  }
  return BS_OK;
}

// Scale tensors as uint32 rows: one row per 128-row block, K/64 tiles of 512
// bytes each; a pair-kernel stage loads two tiles (256 words).
// Scales of the FP4 pair kernel as 8-byte elements, one row per 128-row
// block (K/64 chunks of 512 bytes = K elements); a box is one K stage of `bk`
// elements (bk/64 chunks).
static bs_status sf_map(CUtensorMap* m, const void* sf, int64_t rows, int64_t K, int bk) {
  const uint64_t elems = (uint64_t)K;
  const uint64_t blocks = (uint64_t)((rows + 127) / 128);
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 8, sf, elems, blocks, elems * 8, (uint32_t)bk, 1,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
}

static bs_status launch_fp4(bsk::Fp4Launch& L, const bs_gemm_args* a, int64_t b_rows, int sms, cudaStream_t s,
                            long long pair_tiles, bool grouped) {
  bs_status st;
  L.p.wait_ns = wait_ns(a);
  if (a->fp4_kernel != 1 && sms >= 2) {  // a pair needs two SMs
    const bool split = grouped && a->fp4_small_experts != 2;
    L.p.part = split ? 1 : 0;
    L.p.half_tail = (!grouped && a->fp4_half_tail != 2) ? 1 : 0;
    bsk::Fp4PairLaunch P;
    memset(&P, 0, sizeof P);
    st = fp4_maps(L, a, b_rows, fp4_bk(a));
    if (st != BS_OK) return st;
    st = sf_map(&P.tmSfa, a->sfa, a->M, a->K, fp4_bk(a));
    if (st != BS_OK) return st;
    st = sf_map(&P.tmSfb, a->sfb, b_rows, a->K, fp4_bk(a));
    if (st != BS_OK) return st;
    if (L.epilogue == bsk::kEpiSwiglu || L.epilogue == bsk::kEpiRows ||
        (L.epilogue == bsk::kEpiStore && !grouped)) {
      // boxes of 32 rows x 64 bytes, 64-byte swizzle (32 bytes, 32-byte swizzle
      // for the low-rank variant): the kernel's staging layout
      const bool bf = a->out_dtype == BS_DTYPE_BF16;
      const int es = bf ? 2 : 4;
      const uint32_t row_bytes = L.lora ? 32 : 64;
      st = make_map(&P.tmO, bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, es, a->out,
                    (uint64_t)a->N, (uint64_t)a->M, (uint64_t)a->ldo * es, row_bytes / es, 32,
                    L.lora ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B);
      if (st != BS_OK) return st;
    }
    P.base = L;
    const int pairs = sms / 2;
    P.grid = 2 * (int)(grouped ? pairs : (pair_tiles < pairs ? pair_tiles : pairs));
    cudaError_t e = bsk::launch_fp4_pair_gemm(P, s);
    if (e != cudaSuccess) return cuda_fail(e, "FP4 pair GEMM launch");
    if (split) {
      // the small experts: one CTA per 128-row tile, same operand maps
      L.p.part = 2;
      e = bsk::launch_fp4_gemm(L, s);
      if (e != cudaSuccess) return cuda_fail(e, "FP4 tail GEMM launch");
    }
    return BS_OK;
  }
  st = fp4_maps(L, a, b_rows, fp4_bk(a));
  if (st != BS_OK) return st;
  cudaError_t e = bsk::launch_fp4_gemm(L, s);
  if (e != cudaSuccess) return cuda_fail(e, "FP4 GEMM launch");
  return BS_OK;
}

// Launch plan of an FP8 GEMM: tile width (token columns), tile count, and
// for fewer tiles than SMs the stream-K split: grid G = min(SMs, units), the
// most CTAs sharing one tile (maxc) and the workspace it needs (partials,
// then one counter per tile).
constexpr size_t kStreamKCounterBytes = 4096;

// Stream-K split of `tiles` output tiles of `units` K steps each over at most
// `sms` CTAs: the grid, the most CTAs sharing one tile, and the workspace
// (counter head, then one fp32 partial of 128 x tile_n per share of a tile).
struct SkSplit {
  int grid;
  int maxc;
  size_t ws_bytes;
};
static SkSplit sk_split(long long tiles, long long units, int tile_n, int sms) {
  SkSplit k;
  const long long U = tiles * units;
  const long long G = U < sms ? U : sms;
  k.grid = (int)G;
  k.maxc = 0;
  auto owner = [&](long long u) { return ((u + 1) * G - 1) / U; };
  for (long long t = 0; t < tiles; ++t) {
    const long long n = owner(t * units + units - 1) - owner(t * units) + 1;
    if (n > k.maxc) k.maxc = (int)n;
  }
  k.ws_bytes = kStreamKCounterBytes + (size_t)tiles * (size_t)k.maxc * 128 * (size_t)tile_n * sizeof(float);
  return k;
}

// FP4 decode kernel (M <= 32, swap-AB, stream-K): used unless the caller
// turns it off, there is a low-rank branch, or K is not a multiple of 256.
static bool fp4_decode_applies(const bs_gemm_args* a) {
  return a->fmt == BS_FMT_FP4 && a->M > 0 && a->M <= 32 && !a->lora_t && a->K % 256 == 0 && a->fp4_decode != 2;
}
// Stream-K keeps one arrival counter per tile in the workspace's fixed head.
static bool fp4_decode_stream_k(long long tiles) {
  return tiles <= (long long)(kStreamKCounterBytes / sizeof(int));
}
// CTAs of an FP4 decode launch over `tiles` weight tiles: with at least one
// tile per SM the kernel walks whole tiles, and the 16-token variant, which
// fits two CTAs on an SM, then runs two per SM on the default grid (twice the
// weight bytes in flight); otherwise one per SM.
static int fp4_decode_ctas(const bs_gemm_args* a, long long tiles, int sms) {
  return (a->M <= 16 && a->num_sms == 0 && tiles >= sms) ? 2 * sms : sms;
}

struct Fp8Plan {
  int tile_n;
  long long tiles;
  int grid;
  bool stream_k;
  int maxc;
  size_t ws_bytes, counters_off;  // counters at the start, then the partials
};
static Fp8Plan fp8_plan(const bs_gemm_args* a, int sms, int products = 1) {
  Fp8Plan P;
  memset(&P, 0, sizeof P);
  P.tile_n = bsk::fp8_tile_n(a->M);
  P.tiles = (long long)products * ((a->N + 127) / 128) * ((a->M + P.tile_n - 1) / P.tile_n);
  const long long nkb = a->K / 128;
  P.grid = (int)(P.tiles < sms ? P.tiles : sms);
  P.stream_k = a->fp8_stream_k != 2 && P.tiles < sms && P.tiles <= (long long)(kStreamKCounterBytes / sizeof(int)) &&
               nkb > 1;
  if (!P.stream_k) return P;
  const long long U = P.tiles * nkb;
  const long long G = U < sms ? U : sms;
  P.grid = (int)G;
  auto owner = [&](long long u) { return ((u + 1) * G - 1) / U; };
  for (long long t = 0; t < P.tiles; ++t) {
    const long long n = owner(t * nkb + nkb - 1) - owner(t * nkb) + 1;
    if (n > P.maxc) P.maxc = (int)n;
  }
  // The counters sit in a fixed region at the start of the workspace (one per
  // tile; stream-K runs only with fewer tiles than SMs, so 1024 always
  // suffice) and the partials after it, so calls of different shapes sharing
  // one workspace never find another call's partials where their counters go.
  P.counters_off = 0;
  const size_t parts = (size_t)P.tiles * (size_t)P.maxc * 128 * (size_t)P.tile_n * sizeof(float);
  P.ws_bytes = kStreamKCounterBytes + parts;
  return P;
}

size_t bs_gemm_workspace_bytes(const bs_gemm_args* a) {
  if (!a || a->M <= 0 || a->N <= 0 || a->K < 128 || a->num_sms < 0) return 0;
  int sms = 0;
  if (!device_info(nullptr, &sms)) return 0;
  if (a->num_sms > 0 && a->num_sms < sms) sms = a->num_sms;
  if (fp4_decode_applies(a)) {
    const long long tiles = (a->N + 127) / 128;
    return fp4_decode_stream_k(tiles)
               ? sk_split(tiles, a->K / 256, a->M <= 16 ? 16 : 32, fp4_decode_ctas(a, tiles, sms)).ws_bytes
               : 0;
  }
  if (a->fmt != BS_FMT_FP8) return 0;
  const Fp8Plan P = fp8_plan(a, sms);
  return P.stream_k ? P.ws_bytes : 0;
}

// FP4 decode launch (see fp4_decode_applies) of G >= 1 products that share the
// tokens a->a: product g multiplies by weights b[g] (scales sfb[g]) into
// out[g].  G > 1 takes no per-column scale, bias or weight tensor scale
// (checked by the caller).
static bs_status launch_fp4_decode(const bs_gemm_args* a, int G, const uint8_t* const* b, const uint8_t* const* sfb,
                                   void* const* out, int sms, int* status, cudaStream_t s) {
  bsk::Fp4DecodeLaunch L;
  memset(&L, 0, sizeof L);
  L.tile_n = a->M <= 16 ? 16 : 32;
  const uint64_t kb = (uint64_t)a->K / 2;
  for (int g = 0; g < G; ++g) {
    bs_status st = make_map(G == 1 ? &L.tmW : &L.tmW_g.m[g], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, b[g], kb,
                            (uint64_t)a->N, kb, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != BS_OK) return st;
  }
  bs_status st = make_map(&L.tmX, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a->a, kb, (uint64_t)a->M, kb, 128,
                          (uint32_t)L.tile_n, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != BS_OK) return st;
  bsk::Fp4DecodeParams& p = L.p;
  p.sfw = sfb[0];
  p.sfx = static_cast<const uint8_t*>(a->sfa);
  p.M = (int)a->M;
  p.N = (int)a->N;
  p.K = (int)a->K;
  p.alpha = a->alpha;
  p.col_scale = a->col_scale;
  p.bias = a->bias;
  p.a_ts = a->a_tensor_scale;
  p.b_ts = a->b_tensor_scale;
  p.out = out[0];
  p.out_bf16 = a->out_dtype == BS_DTYPE_BF16;
  p.ldo = a->ldo;
  p.status = status;
  p.wait_ns = wait_ns(a);
  p.pre_b = a->weights_ready == 1 ? bsk::fp4_decode_stages(L.tile_n) : 0;
  p.G = G;
  for (int g = 0; g < G; ++g) {
    p.sfw_g[g] = sfb[g];
    p.out_g[g] = out[g];
  }
  const long long tiles = (long long)G * ((a->N + 127) / 128), units = a->K / 256;
  const int ctas = fp4_decode_ctas(a, tiles, sms);
  if (a->workspace && fp4_decode_stream_k(tiles)) {
    const SkSplit k = sk_split(tiles, units, L.tile_n, ctas);
    if (!aligned16(a->workspace)) return fail(BS_ERR_ALIGN, "workspace must be 16-byte aligned");
    if (a->workspace_bytes < k.ws_bytes)
      return fail(BS_ERR_INVALID, "workspace too small (%zu < %zu bytes)", a->workspace_bytes, k.ws_bytes);
    L.grid = k.grid;
    p.maxc = k.maxc;
    p.counters = static_cast<int*>(a->workspace);
    p.work = reinterpret_cast<float*>(static_cast<uint8_t*>(a->workspace) + kStreamKCounterBytes);
  } else {
    // no workspace (or more tiles than counters): whole tiles only, at least
    // one per CTA
    L.grid = (int)(tiles < ctas ? tiles : ctas);
  }
  cudaError_t e = bsk::launch_fp4_decode(L, s);
  if (e != cudaSuccess) return cuda_fail(e, G == 1 ? "FP4 decode GEMM launch" : "FP4 multi-weight decode launch");
  return BS_OK;
}

// FP8 restrictions shared by bs_gemm and bs_gemm_multi (after check_common).
static bs_status check_fp8(const bs_gemm_args* a) {
  if (a->K % 128) return fail(BS_ERR_ALIGN, "FP8: K=%lld not a multiple of 128", (long long)a->K);
  if (a->alpha != 1.0f || a->col_scale || a->lora_t || a->bias || a->a_tensor_scale || a->b_tensor_scale)
    return fail(BS_ERR_UNSUPPORTED, "FP8 GEMM takes no alpha/col_scale/low-rank/bias/tensor scales");
  if (reinterpret_cast<uintptr_t>(a->sfa) & 3 || reinterpret_cast<uintptr_t>(a->sfb) & 3)
    return fail(BS_ERR_ALIGN, "FP8 scales must be 4-byte aligned");
  return BS_OK;
}

// FP8 launch of G >= 1 products that share the token operand a->a: product g
// multiplies by weights b[g] (scales sfb[g]) into out[g].  G == 1 is bs_gemm's
// kernel; G > 1 the multi-weight variant (one tile list over all products).
// Arguments already checked, M > 0.
static bs_status launch_fp8(const bs_gemm_args* a, int G, const uint8_t* const* b, const float* const* sfb,
                            void* const* out, int sms, int* status, cudaStream_t s) {
  bsk::Fp8Launch L;
  memset(&L, 0, sizeof L);
  L.tile_n = bsk::fp8_tile_n(a->M);
  // swap-AB: the weights [N, K] are the MMA's A operand, the tokens [M, K] its B
  for (int g = 0; g < G; ++g) {
    bs_status st = make_map(G == 1 ? &L.tmA : &L.tmA_g.m[g], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, b[g],
                            (uint64_t)a->K, (uint64_t)a->N, (uint64_t)a->K, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != BS_OK) return st;
  }
  bs_status st = make_map(&L.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a->a, (uint64_t)a->K, (uint64_t)a->M,
                          (uint64_t)a->K, 128, (uint32_t)L.tile_n, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != BS_OK) return st;
  L.p.sfa = static_cast<const float*>(a->sfa);
  L.p.sfb = sfb[0];
  L.p.M = (int)a->M;
  L.p.N = (int)a->N;
  L.p.K = (int)a->K;
  L.p.out = out[0];
  L.p.out_bf16 = a->out_dtype == BS_DTYPE_BF16;
  L.p.ldo = a->ldo;
  L.p.status = status;
  L.p.G = G;
  for (int g = 0; g < G; ++g) {
    L.p.sfb_g[g] = sfb[g];
    L.p.out_g[g] = out[g];
  }
  const Fp8Plan P = fp8_plan(a, sms, G);
  L.p.wait_ns = wait_ns(a);
  L.p.pre_b = a->weights_ready == 1 ? bsk::fp8_stages(P.tile_n) : 0;
  L.p.rowwise = a->fp8_scaling == 2;
  L.grid = P.grid;
  if (P.stream_k && a->workspace) {
    if (!aligned16(a->workspace)) return fail(BS_ERR_ALIGN, "workspace must be 16-byte aligned");
    if (a->workspace_bytes < P.ws_bytes)
      return fail(BS_ERR_INVALID, "workspace too small (%zu < %zu bytes)", a->workspace_bytes, P.ws_bytes);
    L.p.stream_k = 1;
    L.p.maxc = P.maxc;
    L.p.counters = static_cast<int*>(a->workspace);
    L.p.work = reinterpret_cast<float*>(static_cast<uint8_t*>(a->workspace) + kStreamKCounterBytes);
  } else {
    // whole tiles; the 16-token kernel fits two CTAs on an SM, so with at
    // least a tile per SM and the default grid it runs two per SM (twice the
    // weight bytes in flight)
    const int ctas = (P.tile_n == 16 && a->num_sms == 0 && P.tiles >= sms) ? 2 * sms : sms;
    L.grid = (int)(P.tiles < ctas ? P.tiles : ctas);
  }
  cudaError_t e = bsk::launch_fp8_gemm(L, s);
  if (e != cudaSuccess) return cuda_fail(e, G == 1 ? "FP8 GEMM launch" : "FP8 multi-weight GEMM launch");
  return BS_OK;
}

bs_status bs_gemm(const bs_gemm_args* a, bs_stream_t stream) {
  bs_status st = check_common(a, false);
  if (st != BS_OK) return st;
  int* status = nullptr;
  int sms = 0;
  if (!device_info(&status, &sms)) return fail(BS_ERR_CUDA, "no current device");
  if (a->num_sms > 0 && a->num_sms < sms) sms = a->num_sms;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (a->fmt == BS_FMT_FP4) {
    if (a->K % 64) return fail(BS_ERR_ALIGN, "FP4: K=%lld not a multiple of 64", (long long)a->K);
    const bool lora = a->lora_t != nullptr;
    if (lora) {
      if (!a->lora_b_t || a->r != 32) return fail(BS_ERR_INVALID, "low-rank branch needs lora_b_t and r == 32");
      if (a->alpha != 1.0f || a->col_scale)
        return fail(BS_ERR_UNSUPPORTED, "low-rank branch with alpha != 1 or col_scale");
      if (!aligned16(a->lora_t) || !aligned16(a->lora_b_t)) return fail(BS_ERR_ALIGN, "low-rank buffers misaligned");
    }
    if ((a->a_tensor_scale || a->b_tensor_scale) && lora)
      return fail(BS_ERR_UNSUPPORTED, "low-rank branch with two-level tensor scales");
    if ((reinterpret_cast<uintptr_t>(a->a_tensor_scale) | reinterpret_cast<uintptr_t>(a->b_tensor_scale)) & 3)
      return fail(BS_ERR_ALIGN, "tensor scales must be 4-byte aligned");
    if (a->M == 0) return BS_OK;
    if (fp4_decode_applies(a)) {
      const uint8_t* sfb = static_cast<const uint8_t*>(a->sfb);
      void* out = a->out;
      return launch_fp4_decode(a, 1, &a->b, &sfb, &out, sms, status, s);
    }
    bsk::Fp4Launch L;
    memset(&L, 0, sizeof L);
    L.p.sfa = static_cast<const uint8_t*>(a->sfa);
    L.p.sfb = static_cast<const uint8_t*>(a->sfb);
    L.p.M = (int)a->M;
    L.p.N = (int)a->N;
    L.p.K = (int)a->K;
    L.p.alpha = a->alpha;
    L.p.a_ts = a->a_tensor_scale;
    L.p.b_ts = a->b_tensor_scale;
    L.p.col_scale = a->col_scale;
    L.p.bias = a->bias;
    L.p.out = a->out;
    L.p.out_bf16 = a->out_dtype == BS_DTYPE_BF16;
    L.p.ldo = a->ldo;
    L.p.E = 0;
    L.p.status = status;
    L.lora = lora;
    L.epilogue = bsk::kEpiStore;
    const long long tiles = ((a->M + 127) / 128) * ((a->N + 255) / 256);
    L.grid = (int)(tiles < sms ? tiles : sms);
    const long long pair_tiles = ((a->M + 255) / 256) * ((a->N + 255) / 256);
    return launch_fp4(L, a, a->N, sms, s, pair_tiles, false);
  }
  if (a->fmt == BS_FMT_FP8) {
    st = check_fp8(a);
    if (st != BS_OK) return st;
    if (a->M == 0) return BS_OK;
    const uint8_t* b = a->b;
    const float* sfb = static_cast<const float*>(a->sfb);
    void* out = a->out;
    return launch_fp8(a, 1, &b, &sfb, &out, sms, status, s);
  }
  return fail(BS_ERR_INVALID, "fmt %d", a->fmt);
}

size_t bs_gemm_multi_workspace_bytes(const bs_gemm_args* a, int G) {
  if (!a || G < 1 || G > bsk::kMaxProducts || (a->fmt != BS_FMT_FP8 && a->fmt != BS_FMT_FP4) || a->M <= 0 ||
      a->M > 32 || a->N <= 0 || a->K < 128 || a->num_sms < 0)
    return 0;
  int sms = 0;
  if (!device_info(nullptr, &sms)) return 0;
  if (a->num_sms > 0 && a->num_sms < sms) sms = a->num_sms;
  if (a->fmt == BS_FMT_FP4) {
    if (a->K % 256) return 0;
    const long long tiles = (long long)G * ((a->N + 127) / 128);
    return fp4_decode_stream_k(tiles)
               ? sk_split(tiles, a->K / 256, a->M <= 16 ? 16 : 32, fp4_decode_ctas(a, tiles, sms)).ws_bytes
               : 0;
  }
  const Fp8Plan P = fp8_plan(a, sms, G);
  return P.stream_k ? P.ws_bytes : 0;
}

bs_status bs_gemm_multi(const bs_gemm_args* a, int G, const uint8_t* const* b, const void* const* sfb,
                        void* const* out, bs_stream_t stream) {
  if (!a) return fail(BS_ERR_INVALID, "null args");
  if (G < 1 || G > bsk::kMaxProducts) return fail(BS_ERR_INVALID, "G=%d outside [1, %d]", G, bsk::kMaxProducts);
  if (!b || !sfb || !out) return fail(BS_ERR_INVALID, "null weight / scale / output array");
  if (a->fmt != BS_FMT_FP8 && a->fmt != BS_FMT_FP4) return fail(BS_ERR_INVALID, "fmt %d", a->fmt);
  if (a->fmt == BS_FMT_FP8 && a->fp8_scaling == 2)
    return fail(BS_ERR_UNSUPPORTED, "bs_gemm_multi: FP8 block scaling only (not W8A8)");
  if (a->M > 32) return fail(BS_ERR_UNSUPPORTED, "bs_gemm_multi: M=%lld > 32 (decode shapes)", (long long)a->M);
  bs_gemm_args one = *a;
  one.b = b[0];
  one.sfb = sfb[0];
  one.out = out[0];
  bs_status st = check_common(&one, false);
  if (st != BS_OK) return st;
  if (a->fmt == BS_FMT_FP8) {
    st = check_fp8(&one);
    if (st != BS_OK) return st;
  } else {
    if (a->K % 256) return fail(BS_ERR_ALIGN, "bs_gemm_multi FP4: K=%lld not a multiple of 256", (long long)a->K);
    if (a->lora_t || a->col_scale || a->bias || a->b_tensor_scale || a->fp4_decode == 2)
      return fail(BS_ERR_UNSUPPORTED,
                  "bs_gemm_multi FP4: no low-rank branch, col_scale, bias or weight tensor scale; decode kernel only");
    if (reinterpret_cast<uintptr_t>(a->a_tensor_scale) & 3) return fail(BS_ERR_ALIGN, "tensor scale misaligned");
  }
  if (a->M == 0) return BS_OK;
  for (int g = 0; g < G; ++g) {
    if (!b[g] || !sfb[g] || !out[g]) return fail(BS_ERR_INVALID, "null operand of product %d", g);
    if (!aligned16(b[g]) || !aligned16(sfb[g]) || !aligned16(out[g]))
      return fail(BS_ERR_ALIGN, "operands of product %d must be 16-byte aligned", g);
  }
  int* status = nullptr;
  int sms = 0;
  if (!device_info(&status, &sms)) return fail(BS_ERR_CUDA, "no current device");
  if (a->num_sms > 0 && a->num_sms < sms) sms = a->num_sms;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (a->fmt == BS_FMT_FP4)
    return launch_fp4_decode(a, G, b, reinterpret_cast<const uint8_t* const*>(sfb), out, sms, status, s);
  return launch_fp8(a, G, b, reinterpret_cast<const float* const*>(sfb), out, sms, status, s);
}

// FP8 grouped GEMM (tokens as the MMA's M, see gemm_fp8_grouped.cu); args
// already passed check_common.
static bs_status grouped_fp8(const bs_gemm_args* a, int E, const int32_t* offsets, const int32_t* counts,
                             int epilogue, const float* weight_of, cudaStream_t s) {
  if (a->K % 128) return fail(BS_ERR_ALIGN, "FP8: K=%lld not a multiple of 128", (long long)a->K);
  if (epilogue == BS_EPI_COMBINE) return fail(BS_ERR_UNSUPPORTED, "FP8 grouped GEMM: COMBINE epilogue (use ROWS)");
  if (E <= 0 || E > 1024) return fail(BS_ERR_INVALID, "E=%d outside [1, 1024]", E);
  if (!offsets || !counts) return fail(BS_ERR_INVALID, "null offsets/counts");
  if (a->lora_t || a->col_scale || a->bias || a->alpha != 1.0f || a->a_tensor_scale || a->b_tensor_scale ||
      a->fp8_scaling == 2)
    return fail(BS_ERR_UNSUPPORTED, "FP8 grouped GEMM takes no alpha/col_scale/bias/low-rank/tensor scales/W8A8");
  if (epilogue == BS_EPI_SWIGLU && a->out_dtype != BS_DTYPE_BF16) return fail(BS_ERR_INVALID, "SWIGLU output is bf16");
  if (epilogue == BS_EPI_ROWS) {
    if (a->out_dtype != BS_DTYPE_F32) return fail(BS_ERR_INVALID, "ROWS output is fp32");
    if (!weight_of) return fail(BS_ERR_INVALID, "ROWS needs weight_of");
  }
  if (reinterpret_cast<uintptr_t>(a->sfa) & 3 || reinterpret_cast<uintptr_t>(a->sfb) & 3)
    return fail(BS_ERR_ALIGN, "FP8 scales must be 4-byte aligned");
  const int64_t wrows = (epilogue == BS_EPI_SWIGLU ? 2 : 1) * a->N * (int64_t)E;
  if (wrows > (1LL << 30)) return fail(BS_ERR_INVALID, "stacked weights too large");
  const int64_t nbk = epilogue == BS_EPI_SWIGLU ? a->N / (bsk::kFp8GroupedBN / 2)
                                                : (a->N + bsk::kFp8GroupedBN - 1) / bsk::kFp8GroupedBN;
  if ((a->M / 128 + E) * nbk >= (1LL << 31)) return fail(BS_ERR_INVALID, "too many tiles");
  int* status = nullptr;
  int sms = 0;
  if (!device_info(&status, &sms)) return fail(BS_ERR_CUDA, "no current device");
  if (a->num_sms > 0 && a->num_sms < sms) sms = a->num_sms;
  if (a->M == 0) return BS_OK;
  bsk::Fp8GroupedLaunch L;
  memset(&L, 0, sizeof L);
  bs_status st = make_map(&L.tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a->a, (uint64_t)a->K, (uint64_t)a->M,
                          (uint64_t)a->K, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != BS_OK) return st;
  st = make_map(&L.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a->b, (uint64_t)a->K, (uint64_t)wrows, (uint64_t)a->K, 128,
                bsk::kFp8GroupedBN / 2, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != BS_OK) return st;
  L.p.sfa = static_cast<const float*>(a->sfa);
  L.p.sfb = static_cast<const float*>(a->sfb);
  L.p.M = (int)a->M;
  L.p.N = (int)a->N;
  L.p.K = (int)a->K;
  L.p.E = E;
  L.p.offsets = offsets;
  L.p.counts = counts;
  L.p.weight_of = weight_of;
  L.p.out = a->out;
  L.p.out_bf16 = a->out_dtype == BS_DTYPE_BF16;
  L.p.ldo = a->ldo;
  L.p.status = status;
  L.p.wait_ns = wait_ns(a);
  L.epilogue = epilogue == BS_EPI_STORE ? bsk::kEpiStore : epilogue == BS_EPI_SWIGLU ? bsk::kEpiSwiglu : bsk::kEpiRows;
  L.grid = sms;
  cudaError_t e = bsk::launch_fp8_grouped(L, s);
  if (e != cudaSuccess) return cuda_fail(e, "FP8 grouped GEMM launch");
  return BS_OK;
}

bs_status bs_grouped_gemm(const bs_gemm_args* a, int E, const int32_t* offsets, const int32_t* counts,
                          int epilogue, const int32_t* token_of, const float* weight_of, float* out32,
                          int64_t ld_out32, bs_stream_t stream) {
  if (!a) return fail(BS_ERR_INVALID, "null args");
  if (epilogue != BS_EPI_STORE && epilogue != BS_EPI_SWIGLU && epilogue != BS_EPI_COMBINE &&
      epilogue != BS_EPI_ROWS)
    return fail(BS_ERR_INVALID, "epilogue %d", epilogue);
  bs_status st = check_common(a, epilogue == BS_EPI_COMBINE);
  if (st != BS_OK) return st;
  if (a->fmt == BS_FMT_FP8)
    return grouped_fp8(a, E, offsets, counts, epilogue, weight_of, reinterpret_cast<cudaStream_t>(stream));
  if (a->fmt != BS_FMT_FP4) return fail(BS_ERR_INVALID, "fmt %d", a->fmt);
  if (a->K % 64) return fail(BS_ERR_ALIGN, "FP4: K=%lld not a multiple of 64", (long long)a->K);
  if (E <= 0 || E > 1024) return fail(BS_ERR_INVALID, "E=%d outside [1, 1024]", E);
  if (!offsets || !counts) return fail(BS_ERR_INVALID, "null offsets/counts");
  if (a->lora_t || a->col_scale || a->bias || a->alpha != 1.0f || a->a_tensor_scale || a->b_tensor_scale)
    return fail(BS_ERR_UNSUPPORTED, "grouped GEMM takes no alpha/col_scale/bias/low-rank/tensor scales");
  if (epilogue == BS_EPI_SWIGLU && a->out_dtype != BS_DTYPE_BF16) return fail(BS_ERR_INVALID, "SWIGLU output is bf16");
  if (epilogue == BS_EPI_ROWS) {
    if (a->out_dtype != BS_DTYPE_F32) return fail(BS_ERR_INVALID, "ROWS output is fp32");
    if (!weight_of) return fail(BS_ERR_INVALID, "ROWS needs weight_of");
  }
  if (epilogue == BS_EPI_COMBINE) {
    if (!token_of || !weight_of || !out32) return fail(BS_ERR_INVALID, "COMBINE needs token_of, weight_of, out32");
    if (!aligned16(out32) || ld_out32 % 4 || ld_out32 < a->N) return fail(BS_ERR_ALIGN, "out32 misaligned or ld_out32 < N");
  }
  const int64_t wrows = (epilogue == BS_EPI_SWIGLU ? 2 : 1) * a->N * (int64_t)E;
  if (wrows > (1LL << 30)) return fail(BS_ERR_INVALID, "stacked weights too large");
  int* status = nullptr;
  int sms = 0;
  if (!device_info(&status, &sms)) return fail(BS_ERR_CUDA, "no current device");
  if (a->num_sms > 0 && a->num_sms < sms) sms = a->num_sms;
  if (a->M == 0) return BS_OK;
  bsk::Fp4Launch L;
  memset(&L, 0, sizeof L);
  L.p.sfa = static_cast<const uint8_t*>(a->sfa);
  L.p.sfb = static_cast<const uint8_t*>(a->sfb);
  L.p.M = (int)a->M;
  L.p.N = (int)a->N;
  L.p.K = (int)a->K;
  L.p.alpha = 1.0f;
  L.p.out = a->out;
  L.p.out_bf16 = a->out_dtype == BS_DTYPE_BF16;
  L.p.ldo = a->ldo;
  L.p.E = E;
  L.p.offsets = offsets;
  L.p.counts = counts;
  L.p.token_of = token_of;
  L.p.weight_of = weight_of;
  L.p.out32 = out32;
  L.p.ld_out32 = ld_out32;
  L.p.status = status;
  L.p.n_chunk = a->n_chunk_blocks > 0 ? a->n_chunk_blocks : 0;
  L.lora = false;
  L.epilogue = epilogue;
  L.grid = sms;
  return launch_fp4(L, a, wrows, sms, reinterpret_cast<cudaStream_t>(stream), 0, true);
}

bs_status bs_grouped_gemm_swiglu_q4(const bs_gemm_args* a, int E, const int32_t* offsets, const int32_t* counts,
                                    uint8_t* h_codes, uint8_t* h_sf, bs_stream_t stream) {
  if (!a) return fail(BS_ERR_INVALID, "null args");
  if (a->out) return fail(BS_ERR_INVALID, "SWIGLU_Q4 writes h_codes / h_sf: args->out must be NULL");
  bs_status st = check_common(a, true);
  if (st != BS_OK) return st;
  if (a->fmt != BS_FMT_FP4) return fail(BS_ERR_UNSUPPORTED, "SWIGLU_Q4 is FP4 only");
  if (a->K % 64) return fail(BS_ERR_ALIGN, "FP4: K=%lld not a multiple of 64", (long long)a->K);
  if (E <= 0 || E > 1024) return fail(BS_ERR_INVALID, "E=%d outside [1, 1024]", E);
  if (!offsets || !counts) return fail(BS_ERR_INVALID, "null offsets/counts");
  if (a->lora_t || a->col_scale || a->bias || a->alpha != 1.0f || a->a_tensor_scale || a->b_tensor_scale)
    return fail(BS_ERR_UNSUPPORTED, "grouped GEMM takes no alpha/col_scale/bias/low-rank/tensor scales");
  const int64_t wrows = 2 * a->N * (int64_t)E;
  if (wrows > (1LL << 30)) return fail(BS_ERR_INVALID, "stacked weights too large");
  if (a->M > 0) {
    if (!h_codes || !h_sf) return fail(BS_ERR_INVALID, "null h_codes / h_sf");
    if (!aligned16(h_codes) || !aligned16(h_sf)) return fail(BS_ERR_ALIGN, "h_codes / h_sf must be 16-byte aligned");
  }
  int* status = nullptr;
  int sms = 0;
  if (!device_info(&status, &sms)) return fail(BS_ERR_CUDA, "no current device");
  if (a->num_sms > 0 && a->num_sms < sms) sms = a->num_sms;
  if (a->M == 0) return BS_OK;
  bsk::Fp4Launch L;
  memset(&L, 0, sizeof L);
  L.p.sfa = static_cast<const uint8_t*>(a->sfa);
  L.p.sfb = static_cast<const uint8_t*>(a->sfb);
  L.p.M = (int)a->M;
  L.p.N = (int)a->N;
  L.p.K = (int)a->K;
  L.p.alpha = 1.0f;
  L.p.out = h_codes;
  L.p.ldo = a->N / 2;
  L.p.out_sf = h_sf;
  L.p.E = E;
  L.p.offsets = offsets;
  L.p.counts = counts;
  L.p.status = status;
  L.p.n_chunk = a->n_chunk_blocks > 0 ? a->n_chunk_blocks : 0;
  L.lora = false;
  L.epilogue = bsk::kEpiSwigluQ4;
  L.grid = sms;
  return launch_fp4(L, a, wrows, sms, reinterpret_cast<cudaStream_t>(stream), 0, true);
}

bs_status bs_moe_router_topk(const float* logits, int64_t T, int E, int k, int32_t* topk_ids, float* topk_w,
                             bs_stream_t stream) {
  if (T < 0 || E <= 0 || E > 1024) return fail(BS_ERR_INVALID, "router: T=%lld E=%d", (long long)T, E);
  if (k <= 0 || k > E || k > 32) return fail(BS_ERR_INVALID, "router: k=%d outside [1, min(E, 32)]", k);
  if (T > (1LL << 31) / 8) return fail(BS_ERR_INVALID, "router: too many tokens");
  if (T == 0) return BS_OK;
  if (!logits || !topk_ids || !topk_w) return fail(BS_ERR_INVALID, "router: null pointer");
  if ((reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(topk_ids) |
       reinterpret_cast<uintptr_t>(topk_w)) & 3)
    return fail(BS_ERR_ALIGN, "router: buffers must be 4-byte aligned");
  if (!device_info(nullptr, nullptr)) return fail(BS_ERR_CUDA, "no current device");
  cudaError_t e = bsk::launch_moe_router(logits, T, E, k, topk_ids, topk_w, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "router launch");
  return BS_OK;
}

int64_t bs_moe_rows_bound(int64_t T, int k, int E) {
  if (T < 0 || k <= 0 || E <= 0) return 0;
  return T * k + (int64_t)E * 127;
}

size_t bs_moe_dispatch_workspace_bytes(int64_t T, int k, int E) {
  if (T < 0 || k <= 0 || E <= 0) return 0;
  const int64_t P = T * k;
  const int64_t chunks = P > 0 ? (P + 1023) / 1024 : 1;
  return (size_t)chunks * (size_t)E * sizeof(int32_t);
}

bs_status bs_moe_dispatch(const int32_t* topk_ids, const float* topk_w, int64_t T, int k, int E, int32_t* counts,
                          int32_t* offsets, int32_t* pair_of_row, int32_t* token_of, float* weight_of,
                          void* workspace, size_t workspace_bytes, bs_stream_t stream) {
  if (T < 0 || k <= 0 || E <= 0 || E > 1024) return fail(BS_ERR_INVALID, "dispatch: T=%lld k=%d E=%d", (long long)T, k, E);
  if (T * k > (1LL << 30)) return fail(BS_ERR_INVALID, "dispatch: too many pairs");
  if (!counts || !offsets || !pair_of_row || !token_of || !weight_of || !workspace || (T > 0 && (!topk_ids || !topk_w)))
    return fail(BS_ERR_INVALID, "dispatch: null pointer");
  if (workspace_bytes < bs_moe_dispatch_workspace_bytes(T, k, E))
    return fail(BS_ERR_INVALID, "dispatch: workspace too small (%zu < %zu)", workspace_bytes,
                bs_moe_dispatch_workspace_bytes(T, k, E));
  int* status = nullptr;
  if (!device_info(&status, nullptr)) return fail(BS_ERR_CUDA, "no current device");
  cudaError_t e = bsk::launch_moe_dispatch(topk_ids, topk_w, T, k, E, counts, offsets, pair_of_row, token_of,
                                           weight_of, static_cast<int*>(workspace), bs_moe_rows_bound(T, k, E),
                                           status, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "dispatch launch");
  return BS_OK;
}

bs_status bs_moe_dispatch_noalloc(const int32_t* topk_ids, const float* topk_w, int64_t T, int k, int E,
                                  int32_t* counts, int32_t* offsets, int32_t* pair_of_row, int32_t* token_of,
                                  float* weight_of, bs_stream_t stream) {
  if (T < 0 || k <= 0 || E <= 0 || E > 1024) return fail(BS_ERR_INVALID, "dispatch: T=%lld k=%d E=%d", (long long)T, k, E);
  if (T * k > (1LL << 30)) return fail(BS_ERR_INVALID, "dispatch: too many pairs");
  const size_t need = bs_moe_dispatch_workspace_bytes(T, k, E);
  if (need > BS_MOE_DISPATCH_NOALLOC_MAX_BYTES)
    return fail(BS_ERR_INVALID,
                "dispatch_noalloc: T*k=%lld pairs with E=%d need %zu bytes of scratch, above the %u-byte static "
                "array; use bs_moe_dispatch with a caller workspace",
                (long long)(T * k), E, need, (unsigned)BS_MOE_DISPATCH_NOALLOC_MAX_BYTES);
  if (!counts || !offsets || !pair_of_row || !token_of || !weight_of || (T > 0 && (!topk_ids || !topk_w)))
    return fail(BS_ERR_INVALID, "dispatch: null pointer");
  int* status = nullptr;
  if (!device_info(&status, nullptr)) return fail(BS_ERR_CUDA, "no current device");
  cudaError_t e = bsk::launch_moe_dispatch_noalloc(topk_ids, topk_w, T, k, E, counts, offsets, pair_of_row, token_of,
                                                   weight_of, bs_moe_rows_bound(T, k, E), status,
                                                   reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "dispatch_noalloc");
  return BS_OK;
}

bs_status bs_moe_combine(const float* rows, int64_t ld_rows, const int32_t* pair_of_row, int64_t n_rows,
                         int64_t T, int k, int64_t H, int32_t* row_of_pair, void* out, int64_t ldo,
                         bs_stream_t stream) {
  if (T < 0 || n_rows < 0 || H < 0) return fail(BS_ERR_INVALID, "combine: negative size");
  if (k <= 0 || k > 32) return fail(BS_ERR_INVALID, "combine: k=%d outside [1, 32]", k);
  if (T * (int64_t)k > INT32_MAX || n_rows > INT32_MAX) return fail(BS_ERR_INVALID, "combine: too many pairs / rows");
  if (T == 0 || H == 0) return BS_OK;
  if (!rows || !pair_of_row || !row_of_pair || !out) return fail(BS_ERR_INVALID, "combine: null pointer");
  if (H % 8 || ld_rows < H || ld_rows % 4 || ldo < H || ldo % 8)
    return fail(BS_ERR_ALIGN, "combine: H %% 8 == 0, ld_rows >= H (%% 4), ldo >= H (%% 8) required");
  if (!aligned16(rows) || !aligned16(out)) return fail(BS_ERR_ALIGN, "combine: rows / out must be 16-byte aligned");
  if (!device_info(nullptr, nullptr)) return fail(BS_ERR_CUDA, "no current device");
  cudaError_t e = bsk::launch_moe_combine(rows, ld_rows, pair_of_row, n_rows, T, k, H, row_of_pair, out, ldo,
                                          reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  return BS_OK;
}

bs_status bs_moe_finalize(float* out32, void* out_bf16, int64_t n, bs_stream_t stream) {
  if (n < 0) return fail(BS_ERR_INVALID, "finalize: n < 0");
  if (n == 0) return BS_OK;
  if (!out32 || !out_bf16) return fail(BS_ERR_INVALID, "finalize: null pointer");
  if (!aligned16(out32) || !aligned16(out_bf16)) return fail(BS_ERR_ALIGN, "finalize: buffers must be 16-byte aligned");
  if (!device_info(nullptr, nullptr)) return fail(BS_ERR_CUDA, "no current device");
  cudaError_t e = bsk::launch_moe_finalize(out32, out_bf16, n, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "finalize launch");
  return BS_OK;
}

}  // extern "C"
