/*
 * oracle.c -- plain, slow FP64 CPU oracle for block-scaled FP4 / FP8 GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or constant generator with the CUDA path, and the product
 * never calls it.
 *
 * Every function is the plain definition written out: number formats are
 * decoded from their bit-field definitions, encoders are exhaustive nearest
 * searches over the decoded value set, GEMMs are triple loops in double.
 * Threads split output rows only; no blocking, fusion or reordering.
 *
 * Sources (page titles, as cited throughout):
 *   [INFRA]   "Tencent AI Infra interview notes" -- Q "What is FP4
 *             quantization" (format table: E2M1 = 1 sign + 2 exp + 1 mantissa,
 *             16 values, range +-6) and Q "Dimensions and flow of a quantized
 *             matmul" (per-group formula Y = sum_g X_g W_g scale_w[g]).
 *   [W4A4]    "Warp-specialised W4A4 kernel on the newest GPU architecture",
 *             section 1, main formula  Y = (Q(X) Q(W)^T) (.) scale + L(X) + b.
 *   [DG-FP8]  "DeepGEMM teardown (FP8 GEMM)", section 2.1 (e4m3 max 448),
 *             2.2 (per-token / per-block scales), 2.3 (FP32 accumulation),
 *             5.2 (scale = max_val / 448), 5.3 (MoE grouping, contiguous
 *             per-expert rows).
 *   [INFRA-G] "Tencent AI Infra interview notes" -- the scale-granularity
 *             table (per-tensor [1], per-channel [N], per-token [M], per-group)
 *             and W8A8 SmoothQuant: X per-token scale_x [M,1], W per-channel
 *             scale_w [1,N], Y = acc * scale_x * scale_w^T.
 *   [DG-MOE]  "DeepGEMM for Hopper MoE", section 1 (gate -> top-k ->
 *             experts -> weighted sum), section 2.1 (C = TC(A,B) * (sA*sB)),
 *             section 3.1 (fused swish).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* E2M1 ([INFRA] FP4 table): sign bit 3, exponent bits 2..1 (bias 1),
 * mantissa bit 0.  Exponent 0 is subnormal: value = m * 2^-1.  No inf/NaN. */
double orc_e2m1_decode(uint8_t code)
{
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? ldexp((double)m / 2.0, 0)          /* 0.m * 2^(1-1) */
                          : ldexp(1.0 + (double)m / 2.0, e - 1);
    return s ? -mag : mag;
}

/* e4m3fn ([DG-FP8] 2.1: 4 exponent bits, 3 mantissa bits, max finite 448):
 * sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0.  Exponent 0
 * is subnormal (0.m * 2^-6).  S.1111.111 is NaN; there is no infinity. */
double orc_e4m3_decode(uint8_t code)
{
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    double mag = (e == 0) ? ldexp((double)m / 8.0, -6)
                          : ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Round to nearest over the non-negative codes [0, ncodes), ties to the even
 * code (= even mantissa for neighbours), magnitudes above the largest value
 * go to the largest value (saturation).  Exhaustive search. */
static uint8_t nearest_code(double mag, int ncodes, double (*dec)(uint8_t))
{
    /* Saturation: at or above the largest finite value the nearest finite
     * value is that one.  (Tested first: for a magnitude ~2^53 times the
     * maximum every distance below rounds to the same double.) */
    if (mag >= dec((uint8_t)(ncodes - 1)))
        return (uint8_t)(ncodes - 1);
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c < ncodes; ++c) {
        double d = fabs(dec((uint8_t)c) - mag);
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)best;
}

/* Nearest E2M1 code, ties to even, saturating at 6, sign kept (so a negative
 * value that rounds to zero gives code 0b1000). */
uint8_t orc_e2m1_encode(double v)
{
    uint8_t c = nearest_code(fabs(v), 8, orc_e2m1_decode);
    return signbit(v) ? (uint8_t)(c | 8) : c;
}

/* Nearest e4m3fn code, ties to even, saturating at 448 (codes 0..126 are the
 * finite non-negative values), sign kept. */
uint8_t orc_e4m3_encode(double v)
{
    uint8_t c = nearest_code(fabs(v), 127, orc_e4m3_decode);
    return signbit(v) ? (uint8_t)(c | 0x80) : c;
}

/* fp32 correctly rounded quotient a/b of two fp32 values: the double quotient
 * is rounded once more to float; with 53 >= 2*24+2 bits the double rounding is
 * innocuous, so this is IEEE fp32 division. */
static float div_f32(float a, float b) { return (float)((double)a / (double)b); }

/* ------------------------------------------------------------------------ */
/* Quantizers                                                                */
/* ------------------------------------------------------------------------ */

/* FP4 per-group quantization ([INFRA] per-group quantization, group G = 16
 * along K; [W4A4] Q(.)):  per row m and group g of 16 consecutive K elements
 *   amax  = max |x|
 *   s     = e4m3(fl32(amax / 6))                (6 = largest E2M1 value)
 *   code  = e2m1(fl32(x / s)),  or 0 when s == 0
 * x: fp32 [M][ldx]; codes: [M][K/2], element k in the low nibble of byte k/2
 * when k is even, in the high nibble when odd; sf: e4m3 codes [M][K/16].   */
void orc_q4_quantize(const float *x, int64_t M, int64_t K, int64_t ldx,
                     uint8_t *codes, uint8_t *sf)
{
    for (int64_t m = 0; m < M; ++m) {
        const float *row = x + m * ldx;
        for (int64_t g = 0; g < K / 16; ++g) {
            float amax = 0.0f;
            for (int j = 0; j < 16; ++j) {
                float a = fabsf(row[g * 16 + j]);
                if (a > amax) amax = a;
            }
            uint8_t sc = orc_e4m3_encode(div_f32(amax, 6.0f));
            float s = (float)orc_e4m3_decode(sc);
            sf[m * (K / 16) + g] = sc;
            for (int j = 0; j < 16; ++j) {
                int64_t k = g * 16 + j;
                uint8_t c = (s == 0.0f) ? 0 : orc_e2m1_encode(div_f32(row[k], s));
                uint8_t *b = &codes[m * (K / 2) + k / 2];
                if ((k & 1) == 0) *b = (uint8_t)((*b & 0xF0) | c);
                else              *b = (uint8_t)((*b & 0x0F) | (c << 4));
            }
        }
    }
}

/* FP8 quantization with one fp32 scale per block of rows_per_block x 128
 * ([DG-FP8] 2.2 per-token 1x128 activations / 128x128 weight blocks; 5.2
 * scale = max_val / 448):
 *   s    = fl32(amax / 448)
 *   code = e4m3(fl32(x / s)),  or 0 when s == 0
 * x: fp32 [M][ldx]; codes: [M][K]; scales: [ceil(M/rows_per_block)][K/128]. */
void orc_q8_quantize(const float *x, int64_t M, int64_t K, int64_t ldx,
                     int rows_per_block, uint8_t *codes, float *scales)
{
    int64_t nrb = (M + rows_per_block - 1) / rows_per_block;
    for (int64_t rb = 0; rb < nrb; ++rb) {
        int64_t r0 = rb * rows_per_block;
        int64_t r1 = r0 + rows_per_block < M ? r0 + rows_per_block : M;
        for (int64_t kb = 0; kb < K / 128; ++kb) {
            float amax = 0.0f;
            for (int64_t m = r0; m < r1; ++m)
                for (int j = 0; j < 128; ++j) {
                    float a = fabsf(x[m * ldx + kb * 128 + j]);
                    if (a > amax) amax = a;
                }
            float s = div_f32(amax, 448.0f);
            scales[rb * (K / 128) + kb] = s;
            for (int64_t m = r0; m < r1; ++m)
                for (int j = 0; j < 128; ++j) {
                    int64_t k = kb * 128 + j;
                    codes[m * K + k] = (s == 0.0f) ? 0
                                     : orc_e4m3_encode(div_f32(x[m * ldx + k], s));
                }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* GEMMs (threads split output rows)                                          */
/* ------------------------------------------------------------------------ */

typedef struct {
    /* FP4 operands */
    const uint8_t *a, *sfa, *b, *sfb;
    /* FP8 operands */
    const uint8_t *a8, *b8;
    const float *sa8, *sb8;
    int64_t M, N, K;
    double alpha;
    const double *col_scale; /* [N] or NULL */
    const double *t;         /* low-rank left factor T = X A, [M][r] or NULL */
    const double *lb;        /* low-rank right factor B, [r][N] */
    int r;
    const double *bias;      /* [N] or NULL */
    double *y, *s;           /* [M][N] result and error scale sum |terms| */
    int64_t row0, row1;
} gemm_job;

static double e2m1_at(const uint8_t *codes, int64_t rowbytes, int64_t m, int64_t k)
{
    uint8_t byte = codes[m * rowbytes + k / 2];
    return orc_e2m1_decode((k & 1) ? (byte >> 4) : (byte & 15));
}

/* [W4A4] section 1 with [INFRA] per-group dequantization, all in FP64:
 *   y[m,n] = alpha * cs[n] * sum_g sa[m,g] sb[n,g] sum_{k in g} a[m,k] b[n,k]
 *            + sum_r T[m,r] B[r,n] + bias[n]
 *   s[m,n] = |alpha cs[n]| sum_k |sa a sb b| + sum_r |T B| + |bias[n]|      */
static void *fp4_rows(void *p)
{
    gemm_job *j = (gemm_job *)p;
    int64_t G = j->K / 16;
    for (int64_t m = j->row0; m < j->row1; ++m)
        for (int64_t n = 0; n < j->N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t g = 0; g < G; ++g) {
                double sa = orc_e4m3_decode(j->sfa[m * G + g]);
                double sb = orc_e4m3_decode(j->sfb[n * G + g]);
                double part = 0.0, pmag = 0.0;
                for (int64_t k = g * 16; k < g * 16 + 16; ++k) {
                    double prod = e2m1_at(j->a, j->K / 2, m, k) * e2m1_at(j->b, j->K / 2, n, k);
                    part += prod;
                    pmag += fabs(prod);
                }
                acc += part * sa * sb;
                mag += pmag * sa * sb;
            }
            double cs = j->col_scale ? j->col_scale[n] : 1.0;
            double y = j->alpha * cs * acc;
            double s = fabs(j->alpha * cs) * mag;
            if (j->t)
                for (int r = 0; r < j->r; ++r) {
                    double prod = j->t[m * j->r + r] * j->lb[(int64_t)r * j->N + n];
                    y += prod;
                    s += fabs(prod);
                }
            if (j->bias) { y += j->bias[n]; s += fabs(j->bias[n]); }
            j->y[m * j->N + n] = y;
            j->s[m * j->N + n] = s;
        }
    return NULL;
}

/* [DG-MOE] 2.1 and [DG-FP8] 2.2/2.3: per 128-wide K block kb
 *   y[m,n] = sum_kb sa[m,kb] * sb[n/128,kb] * sum_{k in kb} a[m,k] b[n,k]   */
static void *fp8_rows(void *p)
{
    gemm_job *j = (gemm_job *)p;
    int64_t KB = j->K / 128;
    for (int64_t m = j->row0; m < j->row1; ++m)
        for (int64_t n = 0; n < j->N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t kb = 0; kb < KB; ++kb) {
                double sa = j->sa8[m * KB + kb];
                double sb = j->sb8[(n / 128) * KB + kb];
                double part = 0.0, pmag = 0.0;
                for (int64_t k = kb * 128; k < kb * 128 + 128; ++k) {
                    double prod = orc_e4m3_decode(j->a8[m * j->K + k]) *
                                  orc_e4m3_decode(j->b8[n * j->K + k]);
                    part += prod;
                    pmag += fabs(prod);
                }
                acc += part * sa * sb;
                mag += pmag * sa * sb;
            }
            j->y[m * j->N + n] = acc;
            j->s[m * j->N + n] = mag;
        }
    return NULL;
}

static void run_rows(gemm_job *proto, void *(*fn)(void *), int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads > proto->M) nthreads = (int)(proto->M > 0 ? proto->M : 1);
    pthread_t th[256];
    gemm_job jobs[256];
    int64_t per = (proto->M + nthreads - 1) / nthreads;
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = *proto;
        jobs[i].row0 = i * per < proto->M ? i * per : proto->M;
        jobs[i].row1 = (i + 1) * per < proto->M ? (i + 1) * per : proto->M;
        pthread_create(&th[i], NULL, fn, &jobs[i]);
    }
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
}

/* a: codes [M][K/2], sfa: [M][K/16]; b: codes [N][K/2], sfb: [N][K/16];
 * t: [M][r] (may be NULL), lb: [r][N]; y, s: [M][N]. */
void orc_gemm_fp4(const uint8_t *a, const uint8_t *sfa, const uint8_t *b,
                  const uint8_t *sfb, int64_t M, int64_t N, int64_t K,
                  double alpha, const double *col_scale, const double *t,
                  const double *lb, int r, const double *bias, double *y,
                  double *s, int nthreads)
{
    gemm_job j;
    memset(&j, 0, sizeof j);
    j.a = a; j.sfa = sfa; j.b = b; j.sfb = sfb;
    j.M = M; j.N = N; j.K = K; j.alpha = alpha; j.col_scale = col_scale;
    j.t = t; j.lb = lb; j.r = r; j.bias = bias; j.y = y; j.s = s;
    run_rows(&j, fp4_rows, nthreads);
}

/* a8: codes [M][K], sa: [M][K/128]; b8: codes [N][K], sb: [ceil(N/128)][K/128]. */
void orc_gemm_fp8(const uint8_t *a8, const float *sa, const uint8_t *b8,
                  const float *sb, int64_t M, int64_t N, int64_t K, double *y,
                  double *s, int nthreads)
{
    gemm_job j;
    memset(&j, 0, sizeof j);
    j.a8 = a8; j.sa8 = sa; j.b8 = b8; j.sb8 = sb;
    j.M = M; j.N = N; j.K = K; j.y = y; j.s = s;
    run_rows(&j, fp8_rows, nthreads);
}

/* Low-rank left factor of [W4A4] L(X) = X A B, taken on the unquantized X:
 * t[m][r] = sum_k x[m][k] a[k][r], exact in FP64 (x, a hold bf16/fp32 values). */
void orc_lowrank_t(const float *x, int64_t M, int64_t K, int64_t ldx,
                   const float *a, int r, double *t)
{
    for (int64_t m = 0; m < M; ++m)
        for (int j = 0; j < r; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += (double)x[m * ldx + k] * (double)a[k * r + j];
            t[m * r + j] = acc;
        }
}

/* ------------------------------------------------------------------------ */
/* MoE pieces                                                                */
/* ------------------------------------------------------------------------ */

/* Grouping of ([DG-FP8] 5.3): the (token, slot) pairs routed to expert e are
 * stored contiguously, in increasing token order (then slot), and each
 * expert's segment starts on a multiple of `block` rows so that it can be
 * moved in whole blocks.  Outputs:
 *   counts[e]        pairs routed to expert e
 *   offsets[e]       first row of expert e's segment, offsets[E] = total rows
 *   pair_of_row[i]   t*k + slot for a real row, -1 for a padding row
 * pair_of_row must hold offsets[E] entries; the caller sizes it with
 * orc_moe_rows_bound(). */
int64_t orc_moe_rows_bound(int64_t T, int k, int E, int block)
{
    return T * k + (int64_t)E * (block - 1);
}

void orc_moe_dispatch(const int32_t *topk_ids, int64_t T, int k, int E,
                      int block, int32_t *counts, int32_t *offsets,
                      int32_t *pair_of_row)
{
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t p = 0; p < T * k; ++p) counts[topk_ids[p]]++;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) {
        int32_t padded = (counts[e] + block - 1) / block * block;
        offsets[e + 1] = offsets[e] + padded;
    }
    for (int32_t i = 0; i < offsets[E]; ++i) pair_of_row[i] = -1;
    for (int e = 0; e < E; ++e) {
        int32_t row = offsets[e];
        for (int64_t p = 0; p < T * k; ++p)
            if (topk_ids[p] == e) pair_of_row[row++] = (int32_t)p;
    }
}

/* SwiGLU of the gate/up halves ([DG-MOE] 3.1 swish x / (1 + exp(-x))):
 * h = silu(g) * u in FP64.  The caller rounds h to bf16. */
void orc_swiglu(const double *g, const double *u, int64_t n, double *h)
{
    for (int64_t i = 0; i < n; ++i) h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
}

/* Top-k router ([DG-MOE] section 1: the gate's scores pick each token's
 * top-k experts, whose outputs are summed with softmax weights).  For token
 * t the k experts with the largest logits, in descending order of logit,
 * ties going to the lower expert id; weights w[t,j] = exp(l_j - l_0) /
 * sum_i exp(l_i - l_0) over the k chosen logits (l_0 the largest), in FP64.
 * Logits are finite; 1 <= k <= E. */
void orc_moe_router(const float *logits, int64_t T, int E, int k,
                    int32_t *ids, double *w)
{
    unsigned char *taken = (unsigned char *)malloc((size_t)E);
    for (int64_t t = 0; t < T; ++t) {
        const float *l = logits + t * E;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;   /* strict: the lower id keeps a tie */
            }
            taken[best] = 1;
            ids[t * k + j] = best;
        }
        const double top = l[ids[t * k]];
        double sum = 0.0;
        for (int j = 0; j < k; ++j) sum += exp((double)l[ids[t * k + j]] - top);
        for (int j = 0; j < k; ++j) w[t * k + j] = exp((double)l[ids[t * k + j]] - top) / sum;
    }
    free(taken);
}

/* Round a double to the nearest bf16 value (8 significant bits, exponent
 * range of fp32), ties to even, in one step: the significand is scaled to
 * an integer in [128, 256) and rounded with rint() in the default
 * round-to-nearest-even mode.  Values below 2^-126 round to a multiple of
 * 2^-133 (bf16 subnormals); results beyond the largest finite bf16 become
 * infinite.  Returned as a double. */
double orc_round_bf16(double v)
{
    if (v == 0.0 || !isfinite(v)) return v;
    const double a = fabs(v);
    int e;
    frexp(a, &e);                      /* a = f * 2^e, f in [0.5, 1) */
    int q = e - 8;                     /* the unit of the 8th significant bit */
    if (q < -133) q = -133;            /* subnormal spacing */
    const double r = rint(ldexp(a, -q)) * ldexp(1.0, q);
    if (r > 3.3895313892515355e38) return v < 0 ? -INFINITY : INFINITY;
    return v < 0 ? -r : r;
}

/* ------------------------------------------------------------------------ */
/* Format variants                                                           */
/* ------------------------------------------------------------------------ */

/* Two-level FP4 scaling: a per-tensor scale ([INFRA-G] per-tensor row of the
 * granularity table) above the per-group e4m3 scales.  Reading: the tensor
 * scale is the power of two 2^e with the smallest e such that
 * amax_tensor <= 6 * 448 * 2^e, so that the largest group scale
 * amax / (6 * 2^e) fills e4m3's top binade without saturating and applying
 * the tensor scale is exact.  The tensor is divided by 2^e (x' = fl32(x 2^-e))
 * and quantized group by group as orc_q4_quantize does; the value a code
 * stands for is code * s_group * 2^e.  A zero tensor takes e = 0.         */
int orc_q4_two_level_exp(float amax)
{
    if (!(amax > 0.0f)) return 0;
    int e = 0;
    while ((double)amax > 2688.0 * ldexp(1.0, e)) ++e;
    while ((double)amax <= 2688.0 * ldexp(1.0, e - 1)) --e;
    return e;
}

void orc_q4_quantize_two_level(const float *x, int64_t M, int64_t K, int64_t ldx,
                               uint8_t *codes, uint8_t *sf, float *tensor_scale)
{
    float amax = 0.0f;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) {
            float a = fabsf(x[m * ldx + k]);
            if (a > amax) amax = a;
        }
    const int e = orc_q4_two_level_exp(amax);
    float *xs = (float *)malloc((size_t)(M * K > 0 ? M * K : 1) * sizeof(float));
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) xs[m * K + k] = (float)ldexp((double)x[m * ldx + k], -e);
    orc_q4_quantize(xs, M, K, K, codes, sf);
    free(xs);
    *tensor_scale = (float)ldexp(1.0, e);
}

/* FP8 with one fp32 scale per row over all of K ([INFRA-G] W8A8: per-token
 * scale_x [M,1] for activations, per-channel scale_w [1,N] for weights, the
 * weights held as [N, K] so a channel is a row):
 *   s[m]    = fl32(amax_row / 448)
 *   code    = e4m3(fl32(x / s[m])),  or 0 when s[m] == 0                  */
void orc_q8_quantize_rowwise(const float *x, int64_t M, int64_t K, int64_t ldx,
                             uint8_t *codes, float *scales)
{
    for (int64_t m = 0; m < M; ++m) {
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float a = fabsf(x[m * ldx + k]);
            if (a > amax) amax = a;
        }
        const float srow = div_f32(amax, 448.0f);
        scales[m] = srow;
        for (int64_t k = 0; k < K; ++k)
            codes[m * K + k] = (srow == 0.0f) ? 0 : orc_e4m3_encode(div_f32(x[m * ldx + k], srow));
    }
}

/* W8A8 GEMM ([INFRA-G] Y = acc * scale_x * scale_w^T):
 *   y[m,n] = sa[m] * sb[n] * sum_k dec(a[m,k]) dec(b[n,k])   in FP64, and
 *   s[m,n] = sum_k |sa[m] dec(a) sb[n] dec(b)|  (the error scale).        */
void orc_gemm_fp8_rowwise(const uint8_t *a8, const float *sa, const uint8_t *b8,
                          const float *sb, int64_t M, int64_t N, int64_t K,
                          double *y, double *s)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double prod = orc_e4m3_decode(a8[m * K + k]) * orc_e4m3_decode(b8[n * K + k]);
                acc += prod;
                mag += fabs(prod);
            }
            const double f = (double)sa[m] * (double)sb[n];
            y[m * N + n] = f * acc;
            s[m * N + n] = fabs(f) * mag;
        }
}
