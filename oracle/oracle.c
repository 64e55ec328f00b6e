/*
 * CPU oracle for the MoE decode routing path.  TEST INFRASTRUCTURE ONLY:
 * only the tests, the package smoke check and the benchmark's CPU-baseline
 * leg may load it.  It shares no code, header, table or constant generator
 * with the CUDA library; the two meet only through the seeded inputs.
 *
 * Plain, slow and single-threaded on purpose: every function is the written
 * definition of its step, with no blocking, fusion or reordering.  Floating
 * point is fp64 except where the method itself fixes fp32 (the sigmoid score,
 * evaluated in long double and rounded once to fp32, and the selection key
 * of the sigmoid gate, see oracle_sigmoid_f32).
 *
 * Sources (GitHub PR pages about MoE decode routing):
 *  - sglang #36557 "MiniMax-M3: Triton split-K router GEMV with in-kernel
 *    fixup", description: the router GEMV [M,K] bf16 x [N,K] bf16 -> [M,N]
 *    fp32 at N ~ 128, M <= 64.
 *  - sglang #46691 (MiniMax-M3.1 MoE/GEMM kernels), Summary: gate (top-k),
 *    aiter's sort into per-expert blocks, stage-1 activation quant.
 *  - sglang #46652 (Kimi-K3 fused routing/sort/quant), Modifications and the
 *    review diff of the sort kernel: stable rank = number of earlier
 *    (token, slot) pairs on the same expert; MXFP8 stage-1 activations;
 *    896 experts, top-16, hidden 3584.
 * Where the pages are silent (sort layout, MX scale rule, sigmoid rounding,
 * tie order) the readings are stated at each function.
 *
 * Compile with -ffp-contract=off: a fused multiply-add may appear only where
 * it is written as fma()/fmaf().
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* bf16 storage                                                        */
/* ------------------------------------------------------------------ */

static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------ */
/* a1 + a2: router GEMV (split-K is an implementation detail; the      */
/* oracle computes the plain dot products).                            */
/* sglang #36557, description: logits[m, n] = sum_k x[m, k] * W[n, k]. */
/* Products of two bf16 values are exact in fp64; the sum runs in k    */
/* order in fp64 and is rounded once to fp32.                          */
/* ------------------------------------------------------------------ */
void oracle_router_gemv(const uint16_t *x, int64_t ldx, const uint16_t *w,
                        float *logits, int M, int N, int K)
{
    for (int m = 0; m < M; ++m) {
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k)
                acc += bf16_value(x[(int64_t)m * ldx + k]) * bf16_value(w[(int64_t)n * K + k]);
            logits[(int64_t)m * N + n] = (float)acc;
        }
    }
}

/* ------------------------------------------------------------------ */
/* a3: top-k gating.                                                   */
/* ------------------------------------------------------------------ */

/* Order used by every selection: larger key first; equal keys (including
 * +0 and -0, which compare equal) go to the lower expert id. */
typedef struct { float key; int id; } keyed;

static int keyed_cmp(const void *pa, const void *pb)
{
    const keyed *a = (const keyed *)pa, *b = (const keyed *)pb;
    if (a->key > b->key) return -1;
    if (a->key < b->key) return 1;
    return (a->id < b->id) ? -1 : (a->id > b->id);
}

/* Full sort of all N experts by (key desc, id asc); the first k win. */
static void select_topk(const float *key, int N, int k, int32_t *ids_out, keyed *work)
{
    for (int n = 0; n < N; ++n) { work[n].key = key[n]; work[n].id = n; }
    qsort(work, (size_t)N, sizeof(keyed), keyed_cmp);
    for (int j = 0; j < k; ++j) ids_out[j] = work[j].id;
}

/*
 * Softmax gate (MiniMax-style routing: softmax, top-k, renormalise).
 * READING: softmax is monotone, so the top-k of the probabilities is the
 * top-k of the logits; the selection key is the fp32 logit itself, which
 * keeps exp rounding out of the ids.  Weights: the softmax probabilities of
 * the selected experts (fp64), divided by their sum when renormalize != 0.
 */
void oracle_topk_softmax(const float *logits, int M, int N, int k, int renormalize,
                         int32_t *topk_ids, float *topk_weights)
{
    keyed *work = (keyed *)malloc(sizeof(keyed) * (size_t)N);
    double *p = (double *)malloc(sizeof(double) * (size_t)N);
    for (int m = 0; m < M; ++m) {
        const float *l = logits + (int64_t)m * N;
        int32_t *ids = topk_ids + (int64_t)m * k;
        select_topk(l, N, k, ids, work);
        double lmax = -INFINITY;
        for (int n = 0; n < N; ++n) if ((double)l[n] > lmax) lmax = l[n];
        double z = 0.0;
        for (int n = 0; n < N; ++n) { p[n] = exp((double)l[n] - lmax); z += p[n]; }
        for (int n = 0; n < N; ++n) p[n] /= z;
        double s = 0.0;
        for (int j = 0; j < k; ++j) s += p[ids[j]];
        for (int j = 0; j < k; ++j)
            topk_weights[(int64_t)m * k + j] = (float)(renormalize ? p[ids[j]] / s : p[ids[j]]);
    }
    free(p);
    free(work);
}

/*
 * fp32 sigmoid score.  The routing pages fix "fp32 sigmoid scores" for the
 * Kimi-K3-style gate (sglang #46652, Modifications) but not how sigma is
 * evaluated, and two fp32 evaluations that differ by one ulp can swap two
 * experts whose biased scores are one ulp apart.  READING: the score is the
 * plain definition sigma(l) = 1 / (1 + e^-l) of the fp32 logit l, rounded
 * once to the nearest fp32 value (the correctly rounded sigmoid; a tie cannot
 * occur, since sigma of a nonzero rational is irrational).  Evaluated here in
 * long double (a 64-bit significand on x86-64, 113 bits on aarch64), whose
 * relative error of a few 2^-64 is far below the distance of sigma from an
 * fp32 rounding boundary, then rounded once to fp32.  Results below half the
 * smallest fp32 subnormal round to +0; results within 2^-25 of 1 round to 1.
 */
float oracle_sigmoid_f32(float l)
{
    long double e = expl(-(long double)l);
    return (float)(1.0L / (1.0L + e));
}

/* Element-wise oracle_sigmoid_f32 of an array. */
void oracle_sigmoid_f32_array(const float *l, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_sigmoid_f32(l[i]);
}

/*
 * Sigmoid + bias gate (Kimi-K3-style routing).  s_n = sigmoid_f32(l_n); the
 * selection key is t_n = s_n + bias_n in fp32 (bias used for selection only);
 * weights are the unbiased s of the selected experts, divided by their fp64
 * sum when renormalize != 0.  bias may be NULL (treated as zero).
 */
void oracle_topk_sigmoid(const float *logits, const float *bias, int M, int N, int k,
                         int renormalize, int32_t *topk_ids, float *topk_weights)
{
    keyed *work = (keyed *)malloc(sizeof(keyed) * (size_t)N);
    float *s = (float *)malloc(sizeof(float) * (size_t)N);
    float *t = (float *)malloc(sizeof(float) * (size_t)N);
    for (int m = 0; m < M; ++m) {
        const float *l = logits + (int64_t)m * N;
        int32_t *ids = topk_ids + (int64_t)m * k;
        for (int n = 0; n < N; ++n) {
            s[n] = oracle_sigmoid_f32(l[n]);
            t[n] = s[n] + (bias ? bias[n] : 0.0f);
        }
        select_topk(t, N, k, ids, work);
        double sum = 0.0;
        for (int j = 0; j < k; ++j) sum += (double)s[ids[j]];
        for (int j = 0; j < k; ++j)
            topk_weights[(int64_t)m * k + j] =
                (float)(renormalize ? (double)s[ids[j]] / sum : (double)s[ids[j]]);
    }
    free(t);
    free(s);
    free(work);
}

/* ------------------------------------------------------------------ */
/* a4: sort of the (token, slot) assignments into per-expert blocks.   */
/* ------------------------------------------------------------------ */

/*
 * Entries of sorted_token_ids / expert_ids the sort must write, in entries:
 * the worst case of sum_e ceil(c_e / B) * B over all routings, rounded up to
 * a multiple of B: M*k + min(N, M*k) * (B - 1), rounded up to B.
 */
int64_t oracle_sort_capacity(int M, int k, int N, int B)
{
    int64_t mk = (int64_t)M * k;
    int64_t used = mk < N ? mk : N;
    int64_t cap = mk + used * (B - 1);
    return (cap + B - 1) / B * B;
}

/*
 * READING of the sorted layout (the pages name aiter's multi-phase sort but
 * print no layout; the Kimi-K3 sort kernel's review diff gives the stable
 * rank): an assignment is its flat index f = m*k + j.  Experts are laid out
 * in ascending id; within an expert the flat indices ascend (stable); each
 * expert's run is padded to ceil(c_e/B)*B entries with the sentinel M*k, and
 * experts with no assignment get no block.  expert_ids[b] is the expert that
 * owns block b.  Everything past num_tokens_post_padded is filled: sentinel
 * M*k in sorted_token_ids, -1 in expert_ids.  Ids outside [0, N) are not
 * placed (masked experts).  A stable counting sort.
 */
void oracle_moe_sort(const int32_t *topk_ids, int M, int k, int N, int B,
                     int32_t *sorted_token_ids, int32_t *expert_ids,
                     int32_t *num_tokens_post_padded, int64_t capacity)
{
    int64_t mk = (int64_t)M * k;
    int64_t *count = (int64_t *)calloc((size_t)N, sizeof(int64_t));
    int64_t *start = (int64_t *)calloc((size_t)N, sizeof(int64_t));
    int64_t *cursor = (int64_t *)calloc((size_t)N, sizeof(int64_t));
    for (int64_t f = 0; f < mk; ++f) {
        int32_t e = topk_ids[f];
        if (e >= 0 && e < N) count[e]++;
    }
    int64_t pos = 0;
    for (int e = 0; e < N; ++e) {
        start[e] = pos;
        pos += (count[e] + B - 1) / B * B;
    }
    for (int64_t i = 0; i < capacity; ++i) sorted_token_ids[i] = (int32_t)mk;
    for (int64_t b = 0; b < capacity / B; ++b) expert_ids[b] = -1;
    for (int64_t f = 0; f < mk; ++f) {
        int32_t e = topk_ids[f];
        if (e < 0 || e >= N) continue;
        sorted_token_ids[start[e] + cursor[e]] = (int32_t)f;
        cursor[e]++;
    }
    for (int e = 0; e < N; ++e)
        for (int64_t b = start[e] / B; b < (start[e] + (count[e] + B - 1) / B * B) / B; ++b)
            expert_ids[b] = e;
    *num_tokens_post_padded = (int32_t)pos;
    free(cursor);
    free(start);
    free(count);
}

/* ------------------------------------------------------------------ */
/* a5: MXFP8 quantisation (OCP Microscaling Formats v1.0): blocks of   */
/* 32 elements along K share one E8M0 scale; elements are E4M3.        */
/* ------------------------------------------------------------------ */

/*
 * E4M3 (OCP FP8: bias 7, no infinities, max finite 448, smallest subnormal
 * 2^-9) of an exact value v, rounded to nearest with ties to the even code.
 * READING: magnitudes above 448 saturate to +-448 (the MX spec leaves
 * overflow to the implementation; the pages' fp8 producers clamp then round).
 * The sign is kept, so values that round to zero from below give 0x80.
 */
uint8_t oracle_e4m3_encode(double v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (a >= 448.0) return sign | 0x7E;
    if (a < 0x1p-6) {                       /* subnormal range, quantum 2^-9 */
        double q = rint(a * 0x1p9);         /* 0..8; 8 is the smallest normal */
        return sign | (uint8_t)q;
    }
    int e2;
    frexp(a, &e2);                          /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;                         /* floor(log2 a), in [-6, 8] */
    double q = rint(ldexp(a, 3 - e));       /* significand in eighths: 8..16 */
    if (q == 16.0) { q = 8.0; e += 1; }
    return sign | (uint8_t)(((e + 7) << 3) | ((int)q - 8));
}

/* Element-wise e4m3 of an array of exact values (same rounding as above). */
void oracle_e4m3_encode_array(const double *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(v[i]);
}

/*
 * Shared scale of one block: X = floor(log2(amax)) - 8 (8 = emax of E4M3),
 * clamped to [-127, 127]; stored as the E8M0 byte X + 127.  READING: an
 * all-zero block has amax = 0 and takes the lowest scale, X = -127 (byte 0).
 * Elements: e4m3(x * 2^-X).  Output layout: q [M, K] and scale [M, K/32],
 * both row-major in token order.
 */
void oracle_mxfp8_quant(const uint16_t *x, int64_t ldx, int M, int K,
                        uint8_t *q, uint8_t *scale)
{
    for (int m = 0; m < M; ++m) {
        for (int b = 0; b < K / 32; ++b) {
            const uint16_t *blk = x + (int64_t)m * ldx + (int64_t)b * 32;
            double amax = 0.0;
            for (int i = 0; i < 32; ++i) {
                double a = fabs(bf16_value(blk[i]));
                if (a > amax) amax = a;
            }
            int X;
            if (amax == 0.0) {
                X = -127;
            } else {
                int e2;
                frexp(amax, &e2);
                X = (e2 - 1) - 8;
                if (X < -127) X = -127;
                if (X > 127) X = 127;
            }
            scale[(int64_t)m * (K / 32) + b] = (uint8_t)(X + 127);
            for (int i = 0; i < 32; ++i)
                q[(int64_t)m * K + (int64_t)b * 32 + i] = oracle_e4m3_encode(ldexp(bf16_value(blk[i]), -X));
        }
    }
}

/* ------------------------------------------------------------------ */
/* Next row: the router on the norm's scale.                           */
/* sgl-amd-mono #56 page, entry #59 "[Perf] minimax_m31: Run o_proj in */
/* the launch, route on the norm's scale, read B operands from LDS",   */
/* Modifications, "Route on the norm's scale": the RMSNorm in front of */
/* the router hands over each token's rstd, and the router forms the   */
/* normalised activations of its own columns from the un-normalised    */
/* residual sum, so that it sees the norm's output bit for bit.        */
/* READING (the pages print no formula): the norm's output is          */
/*   xn[m, k] = bf16( (x[m, k] * rstd[m]) * s[k] )                     */
/* with both products in fp32, each rounded to nearest even, and       */
/* s[k] = g[k] (plain RMSNorm) or s[k] = 1 + g[k] in fp32 (Gemma       */
/* RMSNorm, the norm the MiniMax-M3 producers of sglang #46691 use,    */
/* "Changes to existing kernels").  bf16 rounding: nearest, ties to    */
/* the even code, as every bf16 store on the pages.                    */
/* ------------------------------------------------------------------ */

/* Nearest bf16 to the finite float f, ties to the even code (the       */
/* definition: compare the distances to the two neighbours exactly).    */
static uint16_t bf16_nearest_even(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t lo = u & 0xFFFF0000u;             /* toward zero, same sign */
    uint32_t hi = lo + 0x10000u;               /* away from zero */
    float flo, fhi;
    memcpy(&flo, &lo, sizeof flo);
    memcpy(&fhi, &hi, sizeof fhi);
    double v = fabs((double)f), a = fabs((double)flo);
    double b = ((hi & 0x7F800000u) == 0x7F800000u) ? 0x1p128 : fabs((double)fhi);
    if (v - a < b - v) return (uint16_t)(lo >> 16);
    if (v - a > b - v) return (uint16_t)(hi >> 16);
    return (uint16_t)((((lo >> 16) & 1u) == 0u) ? (lo >> 16) : (hi >> 16));
}

uint16_t oracle_bf16_round(float f) { return bf16_nearest_even(f); }

void oracle_norm_apply(const uint16_t *x, int64_t ldx, const float *rstd,
                       const uint16_t *g, int gemma, int M, int K, uint16_t *xn)
{
    for (int m = 0; m < M; ++m) {
        for (int k = 0; k < K; ++k) {
            float xv = (float)bf16_value(x[(int64_t)m * ldx + k]);
            float gv = (float)bf16_value(g[k]);
            float s = gemma ? 1.0f + gv : gv;
            float t = xv * rstd[m];
            float p = t * s;
            xn[(int64_t)m * K + k] = bf16_nearest_even(p);
        }
    }
}

/* ------------------------------------------------------------------ */
/* Next row: MXFP4 stage-1 activations.                                */
/* sglang #46691, Summary ("MoE sorting + quant"): the MiniMax-M3.1    */
/* sort kernels quantise the stage-1 activations to MXFP4.  The pages  */
/* give no formula; READING: the OCP Microscaling Formats v1.0 MXFP4   */
/* element and scale rules, laid out like the MXFP8 output.            */
/* ------------------------------------------------------------------ */

/*
 * E2M1 (OCP FP4: 1 sign, 2 exponent bits with bias 1, 1 mantissa bit; no
 * infinities or NaN) of an exact value v: the nearest of the magnitudes
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6 (codes 0..7), ties to the even code;
 * magnitudes above 6 saturate to 6 (READING, as for E4M3).  Sign bit 3 is
 * kept, so values that round to zero from below give 0x8.
 */
uint8_t oracle_e2m1_encode(double v)
{
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    double a = fabs(v);
    if (a >= 6.0) return sign | 0x7;
    int best = 0;
    for (int i = 1; i < 8; ++i) {
        double d = fabs(a - mag[i]), db = fabs(a - mag[best]);
        if (d < db || (d == db && (i & 1) == 0)) best = i;
    }
    return sign | (uint8_t)best;
}

void oracle_e2m1_encode_array(const double *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_encode(v[i]);
}

/*
 * Shared scale of one block of 32: X = floor(log2(amax)) - 2 (2 = emax of
 * E2M1), clamped to [-127, 127]; an all-zero block takes X = -127 (byte 0).
 * Elements: e2m1(x * 2^-X).  Output: q [M, K/2] row-major, two elements a
 * byte, element 2j in the low nibble and 2j + 1 in the high nibble (READING:
 * the usual fp4x2 packing); scale [M, K/32] row-major E8M0 bytes X + 127.
 */
void oracle_mxfp4_quant(const uint16_t *x, int64_t ldx, int M, int K,
                        uint8_t *q, uint8_t *scale)
{
    for (int m = 0; m < M; ++m) {
        for (int b = 0; b < K / 32; ++b) {
            const uint16_t *blk = x + (int64_t)m * ldx + (int64_t)b * 32;
            double amax = 0.0;
            for (int i = 0; i < 32; ++i) {
                double a = fabs(bf16_value(blk[i]));
                if (a > amax) amax = a;
            }
            int X;
            if (amax == 0.0) {
                X = -127;
            } else {
                int e2;
                frexp(amax, &e2);
                X = (e2 - 1) - 2;
                if (X < -127) X = -127;
                if (X > 127) X = 127;
            }
            scale[(int64_t)m * (K / 32) + b] = (uint8_t)(X + 127);
            for (int i = 0; i < 32; i += 2) {
                uint8_t lo = oracle_e2m1_encode(ldexp(bf16_value(blk[i]), -X));
                uint8_t hi = oracle_e2m1_encode(ldexp(bf16_value(blk[i + 1]), -X));
                q[(int64_t)m * (K / 2) + (int64_t)b * 16 + i / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* Next row: stage-1 activations written in sorted order.              */
/* sglang #46691, Summary ("MoE sorting + quant": the sort kernels     */
/* quantise the stage-1 activations) and "Changes to existing          */
/* kernels" (the sort and the stage-1 quant in one launch for decode   */
/* batches).  READING: the grouped expert GEMM reads its A operand     */
/* row by row in the sorted order, so row p of the output, for         */
/* p < num_tokens_post_padded, is the MX quantisation of the token of  */
/* the assignment at sorted position p: x[f / k] with                  */
/* f = sorted_token_ids[p] < M k; a padding position (f = M k) gives   */
/* an all-zero row (codes 0, scale bytes 0: the quantisation of a row  */
/* of zeros).  Rows at or past num_tokens_post_padded are not part of  */
/* the output.  Formats as oracle_mxfp8_quant (fp4 = 0: q [rows, K])   */
/* and oracle_mxfp4_quant (fp4 = 1: q [rows, K/2]); scale [rows, K/32].*/
/* ------------------------------------------------------------------ */
void oracle_sorted_quant(const uint16_t *x, int64_t ldx, int M, int K, int k,
                         const int32_t *sorted_token_ids, int32_t num_tokens_post_padded,
                         int fp4, uint8_t *q, uint8_t *scale)
{
    const int64_t qk = fp4 ? K / 2 : K, sk = K / 32;
    for (int64_t p = 0; p < num_tokens_post_padded; ++p) {
        const int64_t f = sorted_token_ids[p];
        uint8_t *qrow = q + p * qk, *srow = scale + p * sk;
        if (f >= 0 && f < (int64_t)M * k) {
            const uint16_t *xrow = x + (f / k) * ldx;
            if (fp4)
                oracle_mxfp4_quant(xrow, ldx, 1, K, qrow, srow);
            else
                oracle_mxfp8_quant(xrow, ldx, 1, K, qrow, srow);
        } else {
            memset(qrow, 0, (size_t)qk);
            memset(srow, 0, (size_t)sk);
        }
    }
}

/* ------------------------------------------------------------------ */
/* Next row: the shared expert's gate/up projection fused into the     */
/* router launch.  sglang #46691, Summary: the router GEMV's split-K   */
/* partials fuse with the shared expert's fp8 SwiGLU in one launch,    */
/* and the MiniMax-M3.1 shared expert's gate_up is 1536 x 6144;        */
/* sgl-amd-mono #56 page, Modifications: the shared expert runs on     */
/* the checkpoint's MXFP8 values (E4M3 elements, one scale per 32      */
/* along K) with bf16 activations.                                     */
/* ------------------------------------------------------------------ */

/* Exact value of an E4M3 code (OCP FP8: bias 7, subnormals m 2^-9, no
 * infinities; S.1111.111 is NaN). */
double oracle_e4m3_decode(uint8_t c)
{
    const int e = (c >> 3) & 0xF, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    const double v = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return (c & 0x80) ? -v : v;
}

/* bf16 bits of the bf16 value nearest to the finite double v (ties to the
 * even code): the significand at bf16's 8 bits, rint (round to nearest
 * even), subnormals below 2^-126 on the fixed quantum 2^-133. */
uint16_t oracle_bf16_from_double(double v)
{
    const uint16_t sign = signbit(v) ? 0x8000 : 0;
    if (v == 0.0) return sign;
    const double a = fabs(v);
    int e2;
    frexp(a, &e2);
    int ex = e2 - 1;                       /* floor(log2 a) */
    if (ex < -126) ex = -126;
    const double q = rint(ldexp(a, 7 - ex)); /* units of 2^(ex - 7) */
    const float f = (float)ldexp(q, ex - 7); /* exact: at most 9 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)((u >> 16) | sign);
}

/*
 * READING: w13 holds 2I rows of K E4M3 codes, rows [0, I) the gate
 * projection and rows [I, 2I) the up projection (the fused "w13" of a
 * gated MLP), with E8M0 scale bytes w13_scale [2I, K/32]:
 *   W[r, k] = e4m3(w13[r, k]) * 2^(w13_scale[r, k / 32] - 127)
 *   h[m, r] = sum_k x[m, k] W[r, k]                 (fp64, k order)
 *   act[m, i] = silu(h[m, i]) * h[m, I + i],  silu(v) = v / (1 + e^-v)
 * act rounded once to bf16 (nearest even): the input of the shared expert's
 * down projection.  h [M, 2I] is returned as well (the tests derive their
 * tolerance from it).
 */
void oracle_shared_gate_up(const uint16_t *x, int64_t ldx, const uint8_t *w13, const uint8_t *w13_scale,
                           int M, int K, int I, uint16_t *act, double *h)
{
    for (int m = 0; m < M; ++m) {
        for (int r = 0; r < 2 * I; ++r) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k) {
                const double w = ldexp(oracle_e4m3_decode(w13[(int64_t)r * K + k]),
                                       (int)w13_scale[(int64_t)r * (K / 32) + k / 32] - 127);
                acc += bf16_value(x[(int64_t)m * ldx + k]) * w;
            }
            h[(int64_t)m * 2 * I + r] = acc;
        }
        for (int i = 0; i < I; ++i) {
            const double g = h[(int64_t)m * 2 * I + i], u = h[(int64_t)m * 2 * I + I + i];
            act[(int64_t)m * I + i] = oracle_bf16_from_double(g / (1.0 + exp(-g)) * u);
        }
    }
}
