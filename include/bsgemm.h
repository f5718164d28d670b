/*
 * bsgemm.h -- C ABI of the block-scaled FP4 / FP8 GEMM library for GB300
 * (sm_103a).
 *
 * The library computes the block-scaled low-precision matrix multiply
 *
 *     Y = (Q(X) Q(W)^T) (.) scale + L(X) + b
 *
 * ("Warp-specialised W4A4 kernel on the newest GPU architecture", section 1),
 * with Q = FP4 E2M1 codes and one e4m3 scale per 16 consecutive K elements
 * ("Tencent AI Infra interview notes", FP4 format table and per-group
 * quantization), or Q = FP8 e4m3 codes with fp32 scales per 1x128 activation
 * block and per 128x128 weight block ("DeepGEMM teardown (FP8 GEMM)",
 * sections 2.2-2.3), always accumulating in FP32; densely and grouped over
 * MoE experts ("DeepGEMM teardown", section 5.3; "DeepGEMM for Hopper MoE",
 * sections 1 and 3).
 *
 * Conventions shared by every entry point:
 *  - All pointers are DEVICE pointers unless stated otherwise.  The caller
 *    allocates and owns every buffer; the library never allocates, frees or
 *    synchronises.  Calls are asynchronous on `stream` (NULL = legacy stream).
 *  - Matrices are row-major with the K dimension contiguous ("K-major").
 *    Leading dimensions are in elements.
 *  - Host-side validation happens before any launch: a call that returns
 *    anything but BS_OK has launched nothing.
 *  - Device-side failures (a bounded pipeline wait that timed out, an
 *    inconsistent expert-offset table) set a sticky device status word that
 *    bs_get_device_status() reads back; kernels never trap.
 *  - Values are assumed finite.
 */
#ifndef BSGEMM_H
#define BSGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *bs_stream_t; /* same type as cudaStream_t */

typedef enum {
    BS_OK = 0,
    BS_ERR_INVALID = 1,     /* null pointer, bad size or enum value */
    BS_ERR_ALIGN = 2,       /* pointer / leading dimension not 16-byte aligned, K or N not a multiple of the block */
    BS_ERR_UNSUPPORTED = 3, /* valid request this library does not implement */
    BS_ERR_CUDA = 4,        /* a CUDA runtime call failed (launch, attribute, tensor-map encode) */
    BS_ERR_TIMEOUT = 5,     /* device status: a bounded pipeline wait gave up */
    BS_ERR_OFFSETS = 6      /* device status: expert offsets / counts inconsistent */
} bs_status;

typedef enum { BS_DTYPE_F32 = 0, BS_DTYPE_BF16 = 1 } bs_dtype;

typedef enum { BS_FMT_FP4 = 0, BS_FMT_FP8 = 1 } bs_format;

typedef enum {
    BS_EPI_STORE = 0,  /* Y rows written to `out` */
    BS_EPI_SWIGLU = 1, /* grouped only: out[r, n] = bf16(silu(g[r,n]) * u[r,n]) */
    BS_EPI_COMBINE = 2, /* grouped only: out32[token_of[r], n] += weight_of[r] * y[r, n] */
    BS_EPI_ROWS = 3     /* grouped only: out fp32 [r, n] = weight_of[r] * y[r, n] */
} bs_epilogue;

typedef enum {
    BS_Q8_TOKEN_1x128 = 1,     /* one scale per row and 128-wide K block (activations) */
    BS_Q8_BLOCK_128x128 = 128, /* one scale per 128 x 128 block (weights) */
    BS_Q8_ROW = 3              /* one scale per row over all of K (W8A8: per-token activations,
                                  per-channel weights) */
} bs_q8_mode;

/* ---------------------------------------------------------------------------
 * FP4 scale-factor layout ("MMA layout").
 *
 * The e4m3 group scales of an [rows, K] FP4 operand are stored in the order
 * the tensor core reads them: 512-byte tiles, one per (128-row block rb,
 * 64-element K chunk kc), tiles ordered rb-major (tile index rb*(K/64)+kc);
 * inside a tile the scale of row r (0..127) and group j (0..3, 16 elements
 * each) is at byte (r % 32) * 16 + (r / 32) * 4 + j.  Rows are padded to a
 * multiple of 128; padding rows hold zero scales after q4_quantize.
 * ------------------------------------------------------------------------- */

/* Bytes of the scale tensor of an [rows, K] FP4 operand (K % 64 == 0). */
size_t bs_sf_bytes(int64_t rows, int64_t K);

/* Byte offset of the scale of (row, group) where group = k / 16. */
int64_t bs_sf_offset(int64_t row, int64_t group, int64_t K);

/* ---------------------------------------------------------------------------
 * q4_quantize -- FP4 E2M1 group-16 quantization of activations or weights
 * ("Tencent AI Infra interview notes", FP4 format table and per-group
 * quantization; online activation quantization in Q "How does hardware
 * quantize").  For output row i (source row g = gather ? gather[i] : i; a
 * negative g gives an all-zero row) and every group of 16 K elements:
 *     s    = e4m3_rn_satfinite(fl32(amax / 6))
 *     code = e2m1_rn_satfinite(fl32(x / s))     (0 when s == 0)
 * IEEE fp32 division, round to nearest even, saturation at 448 / 6, the sign
 * of a value that rounds to zero is kept (code 0b1000).
 *
 *   x       [*, ldx] fp32 or bf16 (dt); 16-byte aligned, ldx % 8 == 0
 *   M, K    output rows, K % 64 == 0
 *   gather  [M] int32 source-row map, or NULL
 *   codes   [M, K/2] bytes: element k in the low nibble of byte k/2 if k is
 *           even, in the high nibble if odd
 *   sf      bs_sf_bytes(M, K) bytes in the MMA layout above
 *   lora_a_t, r, lora_t (optional, all NULL/0 or all set; bf16 input only):
 *           the left factor of the low-rank branch L(X) = X A B,
 *           T = X A on the UNQUANTIZED rows, with lora_a_t = A^T bf16 [r, K]
 *           (K contiguous) and r == 32.  lora_t receives bf16 [M, 2r]:
 *           columns [0, r) = hi = bf16(T), [r, 2r) = lo = bf16(T - hi), so
 *           hi + lo carries T to about 2^-17 relative.
 * ------------------------------------------------------------------------- */
bs_status q4_quantize(const void *x, bs_dtype dt, int64_t M, int64_t K, int64_t ldx,
                      const int32_t *gather, uint8_t *codes, uint8_t *sf,
                      const void *lora_a_t, int r, void *lora_t, bs_stream_t stream);

/* ---------------------------------------------------------------------------
 * Two-level FP4 scaling: a per-tensor scale above the e4m3 group scales
 * ("Tencent AI Infra interview notes", scale-granularity table: per-tensor,
 * per-channel, per-token, per-group).  The tensor scale is the power of two
 * 2^e with the smallest e such that amax <= 6 * 448 * 2^e; the tensor is
 * divided by it (exactly) and quantized as q4_quantize does, so the largest
 * group scale falls in e4m3's top binade [256, 448] and small weights
 * (N(0, 0.02): one-level group scales are e4m3 subnormals with 2-3
 * significant bits) keep full 3-bit scale mantissas.  A code stands for
 * code * s_group * 2^e; bs_gemm multiplies Y by the two tensor scales
 * (bs_gemm_args.a_tensor_scale / b_tensor_scale).
 *
 * bs_tensor_amax: *amax (device fp32) = max |x| over x [M, K] (K % 8 == 0,
 *   x 16-byte aligned, ldx % 8 == 0).
 * q4_quantize_two_level: codes / sf as q4_quantize (no gather, no low-rank)
 *   of x / 2^e, e from *amax (device, e.g. from bs_tensor_amax); writes
 *   *tensor_scale = 2^e (device fp32).  A zero tensor gets e = 0.
 * ------------------------------------------------------------------------- */
bs_status bs_tensor_amax(const void *x, bs_dtype dt, int64_t M, int64_t K, int64_t ldx, float *amax,
                         bs_stream_t stream);
bs_status q4_quantize_two_level(const void *x, bs_dtype dt, int64_t M, int64_t K, int64_t ldx,
                                const float *amax, uint8_t *codes, uint8_t *sf, float *tensor_scale,
                                bs_stream_t stream);

/* ---------------------------------------------------------------------------
 * bs_fp4_gather_rows -- gather rows of an FP4 matrix that q4_quantize already
 * wrote: output row i = input row gather[i] (a negative or out-of-range index
 * gives a zero row with zero scales), codes copied and each row's scales moved
 * to the output row's place in the MMA scale layout.  Bit-identical to
 * q4_quantize with the same gather on the unquantized rows, because the
 * quantization is row-local; used to group MoE activations by expert
 * ("DeepGEMM teardown", section 5.3) after quantizing each token once.
 *
 *   codes_in, sf_in  [rows_in, K/2] codes and bs_sf_bytes(rows_in, K) scales
 *   gather           int32 [rows_out]
 *   codes_out, sf_out [rows_out, K/2] and bs_sf_bytes(rows_out, K); padding
 *                    rows of the last 128-row block get zero scales
 *   K % 64 == 0, every pointer 16-byte aligned
 * ------------------------------------------------------------------------- */
bs_status bs_fp4_gather_rows(const uint8_t *codes_in, const uint8_t *sf_in, int64_t rows_in, int64_t K,
                             const int32_t *gather, int64_t rows_out, uint8_t *codes_out, uint8_t *sf_out,
                             bs_stream_t stream);

/* ---------------------------------------------------------------------------
 * bs_fp8_gather_rows -- gather rows of an FP8 matrix that q8_quantize wrote in
 * TOKEN (1x128) mode: output row i = input row gather[i] (a negative or
 * out-of-range index gives a zero row with zero scales), codes copied and the
 * row's K-block scales moved to the output row's place.  Bit-identical to
 * q8_quantize of the gathered unquantized rows, because the 1x128 blocks are
 * row-local; groups MoE activations by expert ("DeepGEMM teardown",
 * section 5.3) after quantizing each token once.
 *
 *   codes_in, scales_in    [rows_in, K] e4m3 codes and fp32 [K/128, rows_in]
 *   gather                 int32 [rows_out]
 *   codes_out, scales_out  [rows_out, K] and fp32 [K/128, rows_out]
 *   K % 128 == 0; codes 16-byte aligned, scales 4-byte aligned
 * ------------------------------------------------------------------------- */
bs_status bs_fp8_gather_rows(const uint8_t *codes_in, const float *scales_in, int64_t rows_in, int64_t K,
                             const int32_t *gather, int64_t rows_out, uint8_t *codes_out, float *scales_out,
                             bs_stream_t stream);

/* ---------------------------------------------------------------------------
 * q8_quantize -- FP8 e4m3 quantization with fp32 block scales ("DeepGEMM
 * teardown", section 2.2 per-token / per-block scaling, section 5.2 scale =
 * max_val / 448).  For every block (1 x 128 in BS_Q8_TOKEN_1x128 mode,
 * 128 x 128 in BS_Q8_BLOCK_128x128 mode):
 *     s    = fl32(amax / 448)
 *     code = e4m3_rn_satfinite(fl32(x / s))     (0 when s == 0)
 *
 *   x       [M, ldx] fp32 or bf16; 16-byte aligned, ldx % 8 == 0; K % 128 == 0
 *   codes   [M, K] bytes
 *   scales  TOKEN mode: fp32 [K/128, M] (K-block major: the scales of one K
 *           block are contiguous over rows);
 *           BLOCK mode: fp32 [ceil(M/128), K/128];
 *           ROW mode: fp32 [M] ("Tencent AI Infra interview notes", W8A8
 *           SmoothQuant: scale_x [M, 1] per token, scale_w [1, N] per output
 *           channel, i.e. per row of the [N, K] weights)
 * ------------------------------------------------------------------------- */
bs_status q8_quantize(const void *x, bs_dtype dt, int64_t M, int64_t K, int64_t ldx,
                      int mode, uint8_t *codes, float *scales, bs_stream_t stream);

/* ---------------------------------------------------------------------------
 * bs_gemm -- dense block-scaled GEMM, Y[M, N] = A[M, K] B[N, K]^T.
 *
 * FP4 (fmt = BS_FMT_FP4; "Warp-specialised W4A4 kernel", section 1):
 *     Y[m,n] = alpha * col_scale[n] * sum_g sfa[m,g] sfb[n,g] sum_{k in g} a b
 *              + sum_r T[m,r] Bl[r,n] + bias[n]
 *   a, b       codes [M, K/2] / [N, K/2] as written by q4_quantize
 *   sfa, sfb   bs_sf_bytes(M, K) / bs_sf_bytes(N, K) scale bytes (MMA layout)
 *   alpha      scalar (1 = none); col_scale fp32 [N] or NULL
 *   lora_t     bf16 [M, 2r] hi|lo from q4_quantize, or NULL; lora_b_t =
 *              Bl^T bf16 [N, r]; r == 32.  With lora_t set, alpha must be 1
 *              and col_scale NULL (BS_ERR_UNSUPPORTED otherwise).
 * FP8 (fmt = BS_FMT_FP8; "DeepGEMM for Hopper MoE", section 2.1;
 *      "DeepGEMM teardown", sections 2.2-2.3):
 *     Y[m,n] = sum_kb sa[kb,m] * sb[n/128,kb] * sum_{k in kb} a b  (kb: 128 wide)
 *   a, b       e4m3 codes [M, K] / [N, K]
 *   sfa        fp32 [K/128, M] (q8_quantize TOKEN mode)
 *   sfb        fp32 [ceil(N/128), K/128] (q8_quantize BLOCK mode)
 *   alpha / col_scale / lora / bias must be 1 / NULL / NULL / NULL.
 * Common:
 *   bias       bf16 [N] or NULL (FP4 only)
 *   out        [M, ldo] fp32 or bf16 (out_dtype), 16-byte aligned, ldo % 8 == 0
 *   M >= 0, N % 128 == 0, K % 64 == 0 (FP4) or K % 128 == 0 (FP8)
 *   num_sms    persistent grid size limit (0 = all SMs)
 *   n_chunk_blocks  ignored by bs_gemm (grouped tile-order knob)
 *   fp4_kernel, fp4_stage_k, fp4_small_experts, fp4_half_tail, fp4_decode,
 *   fp8_stream_k, fp8_scaling, wait_timeout_us, weights_ready
 *              per-call kernel choices, described at the fields; 0 = the
 *              library's default.  A zero-initialised struct gets every default.
 *   workspace, workspace_bytes
 *              optional caller-owned device scratch (FP8 and FP4 decode
 *              shapes), see bs_gemm_workspace_bytes.
 * ------------------------------------------------------------------------- */
typedef struct {
    int fmt;                 /* bs_format */
    const uint8_t *a;
    const void *sfa;
    const uint8_t *b;
    const void *sfb;
    int64_t M, N, K;
    float alpha;
    const float *col_scale;
    const void *lora_t;
    const void *lora_b_t;
    int r;
    const void *bias;
    void *out;
    int out_dtype;           /* bs_dtype */
    int64_t ldo;
    int num_sms;
    int n_chunk_blocks;      /* grouped only: tile order walks chunks of this many output
                                column blocks (256 columns; 128 for SWIGLU), all experts per
                                chunk; 0 = one chunk.  Bounds the live out32 slab of COMBINE */
    /* Per-call kernel choices (0 = default).  Other values return BS_ERR_INVALID. */
    int fp4_kernel;          /* FP4: 1 = one CTA per 128 x 256 output tile; 2 = CTA pairs
                                (cta_group::2) on 256 x 256 tiles.  Default: 2 when the call may
                                use two or more SMs, else 1 */
    int fp4_stage_k;         /* FP4: K elements per pipeline stage, 128 or 256 (default 256) */
    int fp4_small_experts;   /* grouped FP4 on CTA pairs: 1 = experts of at most 128 rows run in a
                                second, one-CTA launch (default); 2 = every expert in the pair launch */
    int fp4_half_tail;       /* dense FP4 on CTA pairs: 1 = a last wave that fills at most half of
                                the pairs runs as 256 x 128 half tiles (default); 2 = whole tiles */
    int fp8_stream_k;        /* FP8 with fewer output tiles than SMs (decode shapes): 1 = the
                                tiles' K blocks are shared out evenly over all SMs and the pieces
                                of a tile summed in K order by the last CTA to finish one
                                (stream-K; default, needs `workspace`); 2 = one CTA per tile */
    int fp8_scaling;         /* FP8 scales: 0 or 1 = block-scaled (sfa 1x128 per token, sfb
                                128x128, promoted per 128-wide K block); 2 = W8A8 per row
                                ("Tencent AI Infra interview notes", SmoothQuant): sfa fp32 [M]
                                and sfb fp32 [N] from q8_quantize BS_Q8_ROW,
                                Y = sfa[m] sfb[n] sum_k a b, accumulated over all of K in tensor
                                memory and scaled once */
    int wait_timeout_us;     /* bound of every pipeline wait inside the kernels, in microseconds
                                (default 4,000,000 = 4 s).  A wait that runs out ends the kernel
                                early (outputs undefined) and sets BS_ERR_TIMEOUT in the device
                                status word; it never hangs the GPU */
    int weights_ready;       /* 1 = the kernel launched just before this call on `stream` does not
                                write b or sfb, so the GEMM may start loading them before that
                                kernel has finished (FP8; 0 = wait for it like for every other
                                operand).  Every call is a programmatic dependent launch: its
                                prologue overlaps the tail of the previous kernel on the stream */
    void *workspace;         /* device scratch owned by the caller, 16-byte aligned, of at least
                                bs_gemm_workspace_bytes(args) bytes and ZEROED before its first
                                use; every call leaves it zeroed where the next call reads it.
                                Calls that overlap on the GPU must not share one.  NULL: no
                                scratch (FP8 stream-K then runs one CTA per tile) */
    size_t workspace_bytes;
    const float *a_tensor_scale; /* FP4 dense: device fp32 tensor scales of A and B from
                                    q4_quantize_two_level, or NULL (= 1); Y is multiplied by
                                    both.  Not with the low-rank branch */
    const float *b_tensor_scale;
    int fp4_decode;          /* FP4 with M <= 32 and K % 256 == 0, no low-rank branch: 1 = the
                                decode kernel (swap-AB: weight rows fill the MMA's 128 rows, the
                                tokens its N = 16 or 32; with fewer weight tiles than SMs,
                                stream-K over every SM through `workspace`, else whole
                                tiles; default); 2 = the regular tile kernels */
} bs_gemm_args;

/* Bytes of `workspace` bs_gemm would use for these arguments (sizes, format,
 * num_sms, fp8_stream_k, fp4_decode) on the current device; 0 when it needs
 * none.  Stream-K keeps one arrival counter per tile in the first 4096 bytes (zero
 * between calls) and one fp32 partial tile per CTA share of a tile after
 * them (e.g. M <= 16, N = 7168, K = 4096 on 152 SMs: < 2 MB).  Because the
 * counters always sit at the same place, calls of different shapes may share
 * one workspace as long as they do not overlap on the GPU. */
size_t bs_gemm_workspace_bytes(const bs_gemm_args *args);

bs_status bs_gemm(const bs_gemm_args *args, bs_stream_t stream);

/* ---------------------------------------------------------------------------
 * bs_gemm_multi -- G GEMMs that read one activation, in one launch:
 *     Y_g = A B_g^T,  g = 0 .. G-1,
 * each exactly as bs_gemm computes it for a decode shape (M <= 32): FP8 with
 * block scaling (promotion per 128-wide K block; "DeepGEMM teardown (FP8
 * GEMM)", sections 2.2-2.3), or FP4 through the decode kernel
 * ("Warp-specialised W4A4 kernel", section 1).  The output tiles of all G
 * products form one tile list on one grid, so a decode step's projections of
 * the same tokens pay the launch, first-load and stream-K fix-up latencies
 * that dominate a GEMM with M <= 32 once instead of G times ("DeepGEMM
 * teardown", section 1.2: small M leaves most of the GPU idle; section 3.2:
 * wave scheduling; "Tencent AI Infra interview notes", decode: the GEMM
 * streams its weights, 2KN FLOPs per KN weight bytes).
 *
 *   args      as for bs_gemm with M <= 32; args->a / sfa are the shared
 *             tokens; args->b, sfb and out are ignored; N, K, out_dtype, ldo,
 *             num_sms, fp8_stream_k, weights_ready, wait_timeout_us apply to
 *             every product; the workspace is sized by
 *             bs_gemm_multi_workspace_bytes.
 *             FP8: fp8_scaling 0 or 1 (not W8A8).
 *             FP4: K % 256 == 0; alpha and a_tensor_scale apply to every
 *             product; no low-rank branch, col_scale, bias or b_tensor_scale;
 *             fp4_decode must not be 2.
 *   G         number of products, 1 .. 8
 *   b, sfb, out
 *             HOST arrays of G DEVICE pointers: B_g codes (e4m3 [N, K] or FP4
 *             [N, K/2]), its scales (FP8: fp32 [N/128, K/128] from q8_quantize
 *             BLOCK mode; FP4: bs_sf_bytes(N, K) bytes in the MMA layout), Y_g
 *             [M, ldo]; every pointer 16-byte aligned; the outputs must not
 *             overlap one another or any input
 * Returns BS_ERR_UNSUPPORTED for W8A8, M > 32 or an FP4 option above,
 * BS_ERR_INVALID for G outside [1, 8] or a null array or pointer; otherwise
 * as bs_gemm.
 * ------------------------------------------------------------------------- */
size_t bs_gemm_multi_workspace_bytes(const bs_gemm_args *args, int G);
bs_status bs_gemm_multi(const bs_gemm_args *args, int G, const uint8_t *const *b, const void *const *sfb,
                        void *const *out, bs_stream_t stream);

/* ---------------------------------------------------------------------------
 * bs_grouped_gemm -- FP4 or FP8 GEMM grouped over E experts in one persistent
 * launch ("DeepGEMM teardown", section 1.2 grouped/segmented GEMM and 5.3
 * group offsets; "DeepGEMM for Hopper MoE", section 3 fused expert compute,
 * section 2.1 FP8 expert GEMMs).
 *
 * Rows of A are grouped by expert: expert e owns rows
 * [offsets[e], offsets[e] + counts[e]); every offsets[e] is a multiple of 128
 * and offsets[e+1] >= offsets[e] + counts[e] (bs_moe_dispatch writes such
 * tables).  Expert weights are stacked: B rows [e*Nw, (e+1)*Nw) belong to
 * expert e, with their scales in one bs_sf_bytes(E*Nw, K) tensor; Nw % 128 == 0.
 *
 *   args->a/sfa     A codes / scales for all rows (rows = args->M, the size
 *                   of the grouped buffers, >= offsets[E])
 *   args->b/sfb     stacked expert weights, Nw = 2N (SWIGLU) or N (others)
 *   args->N         output columns per row
 *   offsets, counts device int32 [E+1] / [E]
 *   epilogue        BS_EPI_STORE:   out[r, n] = y (rows r < offsets[e]+counts[e])
 *                   BS_EPI_SWIGLU:  weights rows [0, N) of an expert are the
 *                                   gate, rows [N, 2N) the up projection;
 *                                   out bf16 [M, N] = bf16(silu(g) * u), padding
 *                                   rows of each segment are written as 0
 *                   BS_EPI_COMBINE: out32[token_of[r], n] += weight_of[r] * y[r, n]
 *                                   (fp32 reductions; out32 [*, ld_out32] must
 *                                   be zeroed by the caller or bs_moe_finalize)
 *                   BS_EPI_ROWS:    out fp32 [M, ldo]: out[r, n] = weight_of[r] * y[r, n]
 *                                   for the rows r < offsets[e] + counts[e]; rows
 *                                   past a count may be left unwritten or get
 *                                   weight_of[r] * y[r, n] (bs_moe_dispatch gives
 *                                   them weight 0).  The first half of a
 *                                   two-pass routed combine, see bs_moe_combine
 *   token_of        int32 [M] (COMBINE only); weight_of fp32 [M] (COMBINE, ROWS)
 * Only alpha = 1, no col_scale, no lora and no bias are accepted here.
 *
 * FP8 (args->fmt = BS_FMT_FP8; "DeepGEMM teardown", sections 2.2 and 5.3):
 *   Y[r, n] = sum_kb sa[kb, r] * sb[(e*Nw + n)/128, kb] * sum_{k in kb} a[r,k] b[e*Nw + n, k]
 *   args->a/sfa     e4m3 codes [M, K] and fp32 scales [K/128, M] of all rows
 *                   (q8_quantize TOKEN mode, or bs_fp8_gather_rows)
 *   args->b/sfb     stacked e4m3 weights [E*Nw, K] and their 128x128 block
 *                   scales fp32 [E*Nw/128, K/128] (q8_quantize BLOCK mode of
 *                   the stacked matrix; Nw % 128 == 0, so no block straddles
 *                   two experts)
 *   K % 128 == 0; epilogues STORE, SWIGLU and ROWS as above (COMBINE returns
 *   BS_ERR_UNSUPPORTED); fp8_scaling must not be 2 (W8A8 is dense only).
 * Offsets that break the contract set BS_ERR_OFFSETS in the device status and
 * the kernel writes nothing.
 * ------------------------------------------------------------------------- */
bs_status bs_grouped_gemm(const bs_gemm_args *args, int E, const int32_t *offsets,
                          const int32_t *counts, int epilogue, const int32_t *token_of,
                          const float *weight_of, float *out32, int64_t ld_out32,
                          bs_stream_t stream);

/* ---------------------------------------------------------------------------
 * bs_grouped_gemm_swiglu_q4 -- the SWIGLU grouped GEMM with h re-quantized in
 * its epilogue, so h never goes through memory as bf16 (the "Mega MoE"
 * fusion of "DeepGEMM for Hopper MoE", section 3; FP4 format of the
 * "Warp-specialised W4A4 kernel", section 2).  Same operands and offsets
 * contract as bs_grouped_gemm with BS_EPI_SWIGLU, but args->out must be NULL:
 *   h_codes   uint8 [M, N/2]: the E2M1 codes q4_quantize would write for
 *             h = bf16(silu(g) * u), 16-byte aligned
 *   h_sf      bs_sf_bytes(M, N) bytes: their e4m3 group scales (MMA layout)
 * Rows of each expert's 128-aligned segment are written (padding rows as
 * zero codes and zero scales, like the zero rows of BS_EPI_SWIGLU); rows
 * outside every segment are left untouched.  Bit-identical to BS_EPI_SWIGLU
 * followed by q4_quantize of the segment rows.
 * ------------------------------------------------------------------------- */
bs_status bs_grouped_gemm_swiglu_q4(const bs_gemm_args *args, int E, const int32_t *offsets,
                                    const int32_t *counts, uint8_t *h_codes, uint8_t *h_sf,
                                    bs_stream_t stream);

/* ---------------------------------------------------------------------------
 * bs_moe_router_topk -- top-k routing of every token from its router logits
 * ("DeepGEMM for Hopper MoE", section 1: the gate scores every expert for a
 * token, the top k are chosen and their outputs summed with softmax weights).
 * For token t: topk_ids[t, 0..k) are the k experts with the largest logits in
 * descending order, ties going to the lower expert id (the order a stable sort
 * gives), and topk_w[t, j] = exp(l_j - l_0) / sum_i exp(l_i - l_0) over the k
 * chosen logits, in fp32 (within a few ulp of the exact softmax).
 *
 *   logits    fp32 [T, E], finite; topk_ids int32 [T, k]; topk_w fp32 [T, k]
 *   1 <= E <= 1024, 1 <= k <= min(E, 32); buffers 4-byte aligned
 * The outputs are bs_moe_dispatch's inputs.  Invalid sizes or pointers return
 * BS_ERR_INVALID / BS_ERR_ALIGN before any launch.
 * ------------------------------------------------------------------------- */
bs_status bs_moe_router_topk(const float *logits, int64_t T, int E, int k, int32_t *topk_ids,
                             float *topk_w, bs_stream_t stream);

/* ---------------------------------------------------------------------------
 * bs_moe_dispatch -- group the T*k (token, slot) pairs of a top-k routing by
 * expert ("DeepGEMM teardown", section 5.3: each expert's rows contiguous and
 * movable in whole blocks).  Rows of expert e, in increasing pair index
 * p = t*k + slot, occupy [offsets[e], offsets[e] + counts[e]); offsets[e] is
 * the running sum of counts rounded up to 128.  Unused rows up to
 * bs_moe_rows_bound() get pair -1, token -1 and weight 0.
 *
 *   topk_ids   int32 [T, k], values in [0, E); topk_w fp32 [T, k]
 *   counts     int32 [E];  offsets int32 [E+1]
 *   pair_of_row, token_of int32 [rows_bound]; weight_of fp32 [rows_bound]
 *   workspace  bs_moe_dispatch_workspace_bytes(T, k, E) bytes of device scratch
 * Out-of-range expert ids set BS_ERR_OFFSETS in the device status.
 * ------------------------------------------------------------------------- */
int64_t bs_moe_rows_bound(int64_t T, int k, int E);
size_t bs_moe_dispatch_workspace_bytes(int64_t T, int k, int E);
bs_status bs_moe_dispatch(const int32_t *topk_ids, const float *topk_w, int64_t T, int k,
                          int E, int32_t *counts, int32_t *offsets, int32_t *pair_of_row,
                          int32_t *token_of, float *weight_of, void *workspace,
                          size_t workspace_bytes, bs_stream_t stream);

/* ---------------------------------------------------------------------------
 * bs_moe_dispatch_noalloc -- the same grouping as bs_moe_dispatch, for callers
 * that cannot allocate device memory: a serving runtime that hands out only a
 * fixed memory arena created at start-up, a plugin whose enqueue path must not
 * allocate, or a latency-critical loop where an allocation could synchronise
 * the device.  Such a caller has no place to put bs_moe_dispatch's workspace,
 * so this entry point uses a scratch array that the library itself holds in
 * static device memory; the caller still passes every input and output buffer.
 * The pages have no counterpart of this call.
 *
 *   Arguments, layout and results: as bs_moe_dispatch, minus the workspace.
 *   Limit: bs_moe_dispatch_workspace_bytes(T, k, E) must not exceed
 *          BS_MOE_DISPATCH_NOALLOC_MAX_BYTES (1 MiB; e.g. E = 256 allows up to
 *          1024 chunks of 1024 pairs, T*k <= 1,048,576); larger requests
 *          return BS_ERR_INVALID with a message and launch nothing.
 *   Memory: every GPU that loads the library holds the 1 MiB array until the
 *          process exits.  It calls no cudaMalloc / cudaFree or other
 *          allocating routine.
 *   Set-up: the first call in a CUDA context looks up the array's device
 *          address (cudaGetSymbolAddress, with that context current) and
 *          caches it under the context's unique id; the runtime's primary
 *          context of each device is one such context, and a call from another
 *          context (a driver-API context of the caller's, or a primary
 *          context re-created after cudaDeviceReset) looks the address up
 *          again.  Make the first call in each context before any stream
 *          capture.
 *   Sharing: all calls share the array and it keeps the last call's
 *          contents (each call overwrites everything it reads).  Calls whose
 *          kernels can overlap on the GPU -- different streams or host threads
 *          -- race on it; serialise them.
 * ------------------------------------------------------------------------- */
#define BS_MOE_DISPATCH_NOALLOC_MAX_BYTES (1u << 20)
bs_status bs_moe_dispatch_noalloc(const int32_t *topk_ids, const float *topk_w, int64_t T, int k, int E,
                                  int32_t *counts, int32_t *offsets, int32_t *pair_of_row,
                                  int32_t *token_of, float *weight_of, bs_stream_t stream);

/* bs_moe_finalize -- out[i] = bf16(out32[i]) for n elements, then out32[i] = 0
 * so the accumulator is ready for the next layer call ("DeepGEMM for Hopper
 * MoE", section 3: FP16-class output of the weighted sum). */
bs_status bs_moe_finalize(float *out32, void *out_bf16, int64_t n, bs_stream_t stream);

/* ---------------------------------------------------------------------------
 * bs_moe_combine -- second pass of the two-pass routed combine: the weighted
 * top-k expert outputs of each token are summed into one bf16 row
 * ("Blackwell FP4 MoE TFLOPS optimisation", section 3.2: result aggregation as
 * a stage of its own after the expert matmuls; "DeepGEMM for Hopper MoE",
 * section 3: the weighted sum of the selected experts' outputs).
 *
 *   out[t, n] = bf16( sum over j = 0 .. k-1 of rows[row_of(t, j), n] )
 *
 * summed in fp32 in slot order j (deterministic), where row_of(t, j) is the
 * row bs_moe_dispatch placed pair t*k + j in; pairs the dispatch dropped
 * (out-of-range expert ids) add nothing.
 *
 *   rows         fp32 [n_rows, ld_rows]: weight_of[r] * y[r, :] from
 *                bs_grouped_gemm with BS_EPI_ROWS; 16-byte aligned, ld_rows % 4 == 0
 *   pair_of_row  int32 [n_rows] from bs_moe_dispatch (-1 on padding rows)
 *   T, k, H      tokens, slots per token, columns (H % 8 == 0, H <= ld_rows)
 *   row_of_pair  int32 [T*k] device scratch owned by the caller; written here
 *                (the inverse of pair_of_row, -1 for dropped pairs)
 *   out          bf16 [T, ldo], 16-byte aligned, ldo % 8 == 0, ldo >= H
 * Invalid sizes / pointers return BS_ERR_INVALID or BS_ERR_ALIGN before any launch.
 * ------------------------------------------------------------------------- */
bs_status bs_moe_combine(const float *rows, int64_t ld_rows, const int32_t *pair_of_row, int64_t n_rows,
                         int64_t T, int k, int64_t H, int32_t *row_of_pair, void *out, int64_t ldo,
                         bs_stream_t stream);

/* ---------------------------------------------------------------------------
 * Status.
 * ------------------------------------------------------------------------- */
/* Reads (synchronously) and returns the sticky device status word of the
 * current device: BS_OK, BS_ERR_TIMEOUT or BS_ERR_OFFSETS.  *detail (if not
 * NULL) receives the raw word (error code in the low byte, site id above). */
bs_status bs_get_device_status(int *detail);
/* Resets the device status word of the current device to BS_OK (synchronous). */
bs_status bs_clear_device_status(void);
/* Static description of a status code. */
const char *bs_status_string(bs_status s);
/* Last host-side error message of this thread (after a non-OK return). */
const char *bs_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* BSGEMM_H */
