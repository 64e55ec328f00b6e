/*
 * moe_route.h -- C ABI of the GB300 (sm_103a) MoE decode routing library.
 *
 * The path: a skinny router GEMV (bf16 activations x [M,K] times the bf16 gate
 * W [N,K] -> fp32 logits [M,N]), top-k gating, the sort of the (token, slot)
 * assignments into padded per-expert blocks, and MXFP8 quantisation of the
 * stage-1 activations.  The method follows these GitHub PR pages:
 *   [#36557] sglang "MiniMax-M3: Triton split-K router GEMV with in-kernel
 *            fixup" (description): the GEMV shape, the per-M-bucket split-K
 *            tiling, the in-kernel split-K fixup (the last CTA to finish a
 *            (n-block, row-tile) pair reduces the partials and re-zeroes its
 *            counter slot), and the shape predicate with fall-through.
 *   [#46691] sglang MiniMax-M3.1 MoE/GEMM kernels (Summary; "Changes to
 *            existing kernels"): GEMV up to 512 rows, the gate, aiter's sort
 *            into per-expert blocks, sort + stage-1 quant in one launch for
 *            decode batches, a one-launch decode router for 1-16 tokens that
 *            is bitwise equal to the unfused chain, the int32 offset limit.
 *   [#46652] sglang Kimi-K3 fused MoE routing, sort, quant (Modifications;
 *            Accuracy Tests; review diff of the sort kernel): 896 experts,
 *            top-16, hidden 3584, MXFP8 stage-1 activations, stable ranks.
 *
 * Conventions (all entry points):
 *  - Pointers named x, w, logits, topk_*, sorted_*, expert_ids,
 *    num_tokens_post_padded, q, scale, sel_bias and scratch are DEVICE
 *    pointers owned by the caller.  The library never allocates or frees.
 *  - stream is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Every call is asynchronous on that stream; none synchronises
 *    the host.  The returned status covers argument validation and the launch
 *    (cudaGetLastError) only; a fault inside a kernel surfaces at the
 *    caller's next synchronisation, as for any CUDA call.
 *  - bf16 tensors are row-major with a contiguous last dimension; ldx is the
 *    row stride of x in ELEMENTS.  x, w must be 16-byte aligned and ldx a
 *    multiple of 8; other pointers need their natural alignment.
 *  - All element offsets are computed in 64-bit (no int32 offset limit).
 *  - Validation happens on the host before any launch: a status other than
 *    MR_OK means nothing was launched.  MR_ERR_UNSUPPORTED means the shape is
 *    outside what the kernels cover (the caller may use another path);
 *    MR_ERR_INVALID_ARG means the call itself is wrong.
 *  - Scratch: one caller-owned device buffer per stream, sized by
 *    mr_scratch_bytes() and zeroed ONCE by mr_scratch_reset() (or any
 *    memset) after allocation.  Every successful call leaves its counters
 *    at zero again, so the buffer is reused across launches with no memset.
 *    Two calls that may run concurrently must not share a scratch buffer.
 */
#ifndef MOE_ROUTE_H
#define MOE_ROUTE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MR_ABI_VERSION 2

/* Bytes at the start of every scratch buffer that hold the launch counters. */
#define MR_SCRATCH_COUNTER_BYTES 32768

/* Limits of the kernels (MR_ERR_UNSUPPORTED beyond them). */
#define MR_MAX_EXPERTS 1024
#define MR_MAX_TOPK 32
#define MR_MAX_GEMV_ROWS 512
#define MR_MAX_FUSED_ROWS 64
#define MR_GEMV_K_MULTIPLE 512

typedef enum mr_status {
    MR_OK = 0,
    MR_ERR_UNSUPPORTED = 1,      /* shape / layout outside the kernels' cover  */
    MR_ERR_INVALID_ARG = 2,      /* null or misaligned pointer, bad size       */
    MR_ERR_SCRATCH_TOO_SMALL = 3,/* scratch_bytes below what the call needs    */
    MR_ERR_CUDA = 4,             /* the CUDA runtime reported an error         */
    MR_ERR_TIMEOUT = 5,          /* mr_device_error: a bounded wait ran out    */
    MR_ERR_SCRATCH_DIRTY = 6     /* debug check: scratch counters not zero     */
} mr_status;

typedef enum mr_scoring {
    MR_SCORE_SOFTMAX = 0,        /* select by logit; weights = softmax         */
    MR_SCORE_SIGMOID = 1         /* select by sigmoid + bias; weights = sigmoid */
} mr_scoring;

typedef enum mr_norm_kind {
    MR_NORM_RMS = 0,             /* RMSNorm: scale = g                         */
    MR_NORM_GEMMA = 1            /* Gemma RMSNorm: scale = 1 + g (fp32)        */
} mr_norm_kind;

typedef enum mr_quant_format {
    MR_QUANT_NONE = 0,           /* no stage-1 activation quant               */
    MR_QUANT_MXFP8 = 1,          /* E4M3 codes q [M, K], E8M0 scales [M, K/32] */
    MR_QUANT_MXFP4 = 2           /* E2M1 codes q [M, K/2], E8M0 scales [M, K/32] */
} mr_quant_format;

/* Launch options, process-wide (bits for mr_set_launch_flags). */
#define MR_LAUNCH_PDL 1         /* programmatic dependent launch, see below */
#define MR_LAUNCH_TEST_STALL 2  /* test hook for the timeout path, see below */
#define MR_LAUNCH_LEGACY_MMA 4  /* router GEMV on mma.sync instead of tcgen05 */
#define MR_LAUNCH_TEST_SLOW_SIGMOID 8  /* test hook: exact sigmoid always by its slow path */
#define MR_LAUNCH_CHECK_SCRATCH 16   /* debug: verify scratch counters before a launch */

/*
 * Sets the launch options of every later call in this process; returns
 * MR_ERR_INVALID_ARG for unknown bits.  With MR_LAUNCH_PDL each kernel is
 * launched with programmatic stream serialization: it may start while the
 * kernel before it on the stream is still running, issues its loads of the
 * gate weight w at once, and waits for that kernel to complete before it
 * touches anything else (x, logits, ids, scratch, outputs).  The caller must
 * then not write w in the kernel launched just before the routing call on
 * the same stream.  With MR_LAUNCH_LEGACY_MMA the router GEMV of more than
 * 64 rows runs as the split-K GEMV with last-arriver fixup on warp-level
 * mma.sync instead of the tcgen05 cluster kernel (the two sum the split-K
 * partials in different orders, so their logits agree within fp32 rounding,
 * not bit for bit); up to 64 rows it always runs on mma.sync.
 * MR_LAUNCH_TEST_SLOW_SIGMOID (a test of the sigmoid gate, never for
 * production): every exact sigmoid score takes its double-double path
 * instead of the fp64 fast path with its rounding test; the outputs are the
 * same bits, only slower.
 * MR_LAUNCH_CHECK_SCRATCH (a debug check): a call that is about to launch a
 * kernel that uses the scratch counters (the split-K GEMV's last-arriver
 * fixup [#36557 description: the last CTA re-zeroes its counter slot], the
 * sort of more than 2048 assignments, the one-launch route over several
 * clusters or expert groups) first copies the counter prefix to the host on
 * its stream and waits for it; if any counter is not zero (a scratch buffer
 * that was never zeroed, was written by someone else, or is in use by a
 * call on another stream) it returns MR_ERR_SCRATCH_DIRTY and launches
 * nothing.  It makes those calls synchronous: do not use it under stream
 * capture or in production.
 * Default: 0 (plain stream order, tcgen05 where the weight tile fits).
 */
int mr_set_launch_flags(int flags);
int mr_get_launch_flags(void);

/*
 * Bounded waits.  The router GEMV for M <= 64 and the one-launch route hand
 * data between the CTAs of a thread-block cluster (split-K partials to the
 * CTA that owns a token, chosen ids to the CTA that sorts).  Each receiving
 * CTA waits for the bytes it expects at most the wait limit (default 1 s).
 * When a wait runs out the kernel sets a device-side flag and returns early;
 * the outputs of that call are undefined, and after a call with M > 16 the
 * scratch counters must be zeroed again (mr_scratch_reset).
 * mr_set_wait_limit_ns: 1e3 <= ns <= 6e10, else MR_ERR_INVALID_ARG;
 * process-wide, for later calls.
 * mr_device_error: MR_ERR_TIMEOUT if a wait ran out on the current device
 * since the flag was last cleared, else MR_OK (MR_ERR_CUDA if the flag could
 * not be read); clear != 0 also clears it.  Synchronous: call it after the
 * routing calls' streams have finished.
 * MR_LAUNCH_TEST_STALL (a test of this path, never for production): every
 * receiving CTA expects 16 bytes more than are sent, so its wait runs out.
 */
int mr_set_wait_limit_ns(uint64_t ns);
int mr_device_error(int clear);

/* Human-readable name of a status code (static string, never NULL). */
const char *mr_status_string(int status);

/* The cudaError_t value behind the calling thread's most recent
 * MR_ERR_CUDA (0 when no call of this thread has returned MR_ERR_CUDA). */
int mr_last_cuda_error(void);

/* MR_ABI_VERSION of the loaded library. */
int mr_abi_version(void);

/*
 * Shape predicate of the router GEMV [#36557 description: "router_gemv_
 * supported()": dtype, contiguous last dim, N % BLOCK_N, K % BLOCK_K, M].
 * Returns 1 when mr_router_gemv covers (M, N, K, ldx), else 0.  Pure host
 * function.  Covered: 1 <= M <= 512, 8 <= N <= 1024 with N divisible by the
 * bucket's n-block, K a positive multiple of 512, ldx >= K and ldx % 8 == 0.
 */
int mr_router_gemv_supported(int M, int N, int K, int64_t ldx);

/*
 * Scratch bytes sufficient for every call of this library with M <= M_max
 * tokens, N experts, hidden K and top-k (router GEMV split-K partials of
 * either kernel above 64 rows, the fused route, the multi-CTA sort of large
 * batches).  The first
 * MR_SCRATCH_COUNTER_BYTES hold counters.  Returns 0 for out-of-range
 * arguments.  Pure host function.
 */
size_t mr_scratch_bytes(int M_max, int N, int K, int topk);

/* Zeroes scratch[0, scratch_bytes) on stream (one cudaMemsetAsync). */
int mr_scratch_reset(void *scratch, size_t scratch_bytes, void *stream);

/*
 * a1 + a2. Router GEMV with in-kernel split-K fixup [#36557 description;
 * #46691 Summary: up to 512 rows].
 *   logits[m, n] = sum_k x[m, k] * w[n, k]   (fp32 accumulation)
 * x: bf16 [M, ldx]; w: bf16 [N, K] contiguous; logits: fp32 [M, N].
 * One launch.  The K range is split over CTAs and the partials are summed in
 * split order (deterministic: the same inputs give the same bits on every
 * call):
 *  - M <= 64 when the cluster kernel's tiles fit: one thread-block cluster
 *    per 16 rows, each CTA a K slice, the partials summed by each row's
 *    owner CTA over distributed shared memory; no scratch.  The experts are
 *    split into groups (one cluster each) as far as the co-resident
 *    clusters allow.  These are the logits of mr_moe_route_sort_quant, bit
 *    for bit;
 *  - 64 < M <= 512 with N <= 128 (and K / cluster size a multiple of 16, at
 *    most 8 stages of 64): the tensor-core GEMV (tcgen05, one cluster per
 *    group of rows, each CTA a K slice); its partials pass through the
 *    scratch work area (mr_scratch_bytes covers them), so it runs only
 *    with a scratch of at least that size;
 *  - otherwise the split-K kernel: the last CTA to finish each (n-block,
 *    row-tile) sums the fp32 partials and re-zeroes its counter (scratch
 *    of mr_scratch_bytes bytes, else MR_ERR_INVALID_ARG / _SCRATCH_TOO_SMALL).
 */
int mr_router_gemv(const void *x, int64_t ldx, const void *w, float *logits,
                   int M, int N, int K, void *scratch, size_t scratch_bytes,
                   void *stream);

/*
 * a3. Top-k gating [#46691 Summary: the gate; #46652: sigmoid gate with a
 * selection bias, top-16 of 896].  One warp per token.
 *   MR_SCORE_SOFTMAX: selection key = the logit; weights = softmax
 *     probabilities of the selected experts (divided by their sum when
 *     renormalize != 0).
 *   MR_SCORE_SIGMOID: s = sigmoid(logit) = 1 / (1 + e^-logit) rounded once
 *     to the nearest fp32 value (correctly rounded: an fp64 evaluation with a
 *     rounding test, double-double where that test cannot decide); key =
 *     s + sel_bias[n] in fp32; weights = the unbiased s of the selected
 *     (divided by their sum when renormalize != 0).  Only experts whose fp32
 *     approximate key is near the k-th largest are scored exactly; the ids
 *     are those of the exact keys.
 * Ties: the lower expert id wins; -0 and +0 tie.  Slot j of a token is its
 * j-th best expert.  logits: fp32 [M, N]; sel_bias: fp32 [N] or NULL
 * (sigmoid only); topk_ids: int32 [M, topk]; topk_weights: fp32 [M, topk].
 * Requires 1 <= topk <= min(N, 32).  NaN logits are outside the contract.
 */
int mr_route_topk(const float *logits, int M, int N, int topk, int scoring,
                  const float *sel_bias, int renormalize, int32_t *topk_ids,
                  float *topk_weights, void *stream);

/*
 * Entries the sort writes into sorted_token_ids: the worst case of
 * sum_e ceil(c_e / block) * block, i.e. M*topk + min(N, M*topk)*(block-1),
 * rounded up to a multiple of block.  expert_ids holds capacity / block
 * entries.  Returns -1 for out-of-range arguments.  Pure host function.
 */
int64_t mr_sort_capacity(int M, int topk, int N, int block);

/*
 * a4. Sort of the assignments into padded per-expert blocks [#46691 Summary
 * and "Changes to existing kernels": aiter's sort; #46652 review diff: the
 * stable rank of an assignment is the number of earlier (token, slot) pairs
 * on the same expert].
 * Layout: assignment f = m*topk + j.  Experts in ascending id; within an
 * expert, f ascending; each expert's run padded to a multiple of block with
 * the sentinel M*topk; experts with no assignment take no block.
 * expert_ids[b] = the expert owning block b.  *num_tokens_post_padded = the
 * padded total.  Every entry past it, up to capacity (resp. capacity/block),
 * is written: sentinel M*topk (resp. -1).  Ids outside [0, N) are not placed.
 * topk_ids: int32 [M, topk]; sorted_token_ids: int32 [capacity];
 * expert_ids: int32 [capacity / block]; num_tokens_post_padded: int32 [1].
 * capacity must be >= mr_sort_capacity(M, topk, N, block).  1 <= block <=
 * 1024.  One launch up to 65536 assignments (over up to one CTA per SM, each
 * CTA counting every id and placing the assignments of its own token rows;
 * scratch unused, may be NULL); two launches above (scratch used).  Output
 * bits are unique (no freedom in the layout).
 */
int mr_moe_sort(const int32_t *topk_ids, int M, int topk, int N, int block,
                int32_t *sorted_token_ids, int32_t *expert_ids,
                int32_t *num_tokens_post_padded, int64_t capacity,
                void *scratch, size_t scratch_bytes, void *stream);

/*
 * a5. MXFP8 quantisation of the stage-1 activations [#46691 Summary: sort +
 * stage-1 activation quant; #46652 Accuracy Tests: MXFP8], per the OCP
 * Microscaling Formats v1.0 spec: for each row and block of 32 elements
 * along K, X = floor(log2(amax)) - 8, clamped to [-127, 127] (amax = 0 gives
 * -127); scale[m, b] = X + 127 (E8M0); q = E4M3(x * 2^-X), round to nearest
 * even, saturating to +-448, sign kept.  Exact (no fast-math): bf16
 * subnormals are honoured.  x: bf16 [M, ldx]; q: uint8 [M, K] row-major;
 * scale: uint8 [M, K/32] row-major.  K % 32 == 0.  Any M >= 1.
 */
int mr_mxfp8_quant(const void *x, int64_t ldx, int M, int K, uint8_t *q,
                   uint8_t *scale, void *stream);

/*
 * a6. The whole path for 1 <= M <= 64 tokens in ONE launch [#46691 Summary:
 * a one-launch decode router for 1-16 tokens, bitwise equal to router GEMV,
 * gate and sort; sort + quant in one launch for decode batches].
 * Arguments as in the four calls above; every output is bitwise equal to
 * mr_router_gemv -> mr_route_topk -> mr_moe_sort -> mr_mxfp8_quant on the
 * same inputs.  q and scale may both be NULL to skip the quantisation.
 * K % 512 == 0, N % 8 == 0, N <= 1024, topk <= 32.
 * One thread-block cluster per 16 tokens.  M <= 16 needs no scratch (scratch
 * may be NULL).  M > 16: the clusters hand over through scratch by an atomic
 * last-arriver ticket (no spin-waits) and the last cluster sorts; scratch
 * must hold mr_scratch_bytes(M, N, K, topk) bytes (MR_ERR_INVALID_ARG if
 * NULL, MR_ERR_SCRATCH_TOO_SMALL if short).
 * Many experts (N >= 512) with M <= 16: given a scratch of
 * mr_scratch_bytes(M, N, K, topk) bytes, the experts are split into groups of
 * >= 128, one cluster each, so that more SMs share the gate weight; each
 * cluster's top-k candidates per token go through scratch to the cluster
 * that takes the last ticket, which merges them and sorts.  Without that
 * scratch the route runs unsplit.  The outputs are the same bits either way.
 */
int mr_moe_route_sort_quant(const void *x, int64_t ldx, const void *w,
                            int M, int N, int K, int topk, int scoring,
                            const float *sel_bias, int renormalize, int block,
                            float *logits, int32_t *topk_ids, float *topk_weights,
                            int32_t *sorted_token_ids, int32_t *expert_ids,
                            int32_t *num_tokens_post_padded, int64_t capacity,
                            uint8_t *q, uint8_t *scale,
                            void *scratch, size_t scratch_bytes, void *stream);

/*
 * a4 + a5 in ONE launch for decode batches [#46691 Summary: the MiniMax-M3.1
 * sort and stage-1 quant run as one launch for decode batches and as four
 * launches for prefill].  The sort outputs are bitwise equal to mr_moe_sort.
 * The quantisation, exactly as mr_mxfp8_quant (quant_format MR_QUANT_MXFP8)
 * or mr_mxfp4_quant (MR_QUANT_MXFP4), is written
 *  - in token order: q [M, K] (MXFP8) or [M, K/2] (MXFP4), scale [M, K/32],
 *    bitwise equal to those calls; or
 *  - with MR_QUANT_SORTED_ROWS or-ed into quant_format, in sorted order for
 *    the grouped expert GEMM [#46691 Summary "MoE sorting + quant"]: q has
 *    capacity rows of K (MXFP8) or K/2 (MXFP4) bytes and scale capacity rows
 *    of K/32 bytes; for p < *num_tokens_post_padded, row p is the
 *    quantisation of x[sorted_token_ids[p] / topk] and a padding position
 *    (sentinel M*topk) is a row of zero codes and zero scale bytes.  Rows at
 *    or past *num_tokens_post_padded are not written.
 * Arguments and layouts as there; x is bf16 [M, ldx] with the rows of
 * topk_ids.  One launch over up to one CTA per SM, no scratch.
 * M * topk <= MR_SORT_QUANT_MAX_ASSIGN (8192 tokens at top-8) and K % 32 == 0,
 * else MR_ERR_UNSUPPORTED; MR_QUANT_NONE or an unknown format, a NULL or
 * misaligned (8 B) q, or a NULL scale returns MR_ERR_INVALID_ARG.
 */
#define MR_SORT_QUANT_MAX_ASSIGN 65536
#define MR_QUANT_SORTED_ROWS 0x100
int mr_moe_sort_quant(const int32_t *topk_ids, int M, int topk, int N, int block,
                      const void *x, int64_t ldx, int K, int quant_format,
                      int32_t *sorted_token_ids, int32_t *expert_ids,
                      int32_t *num_tokens_post_padded, int64_t capacity,
                      uint8_t *q, uint8_t *scale, void *stream);

/*
 * a5, MXFP4 variant [sglang #46691 Summary: the MiniMax-M3.1 sort kernels
 * MXFP4-quantise the stage-1 activations], per the OCP Microscaling Formats
 * v1.0 spec: for each row and block of 32 elements along K,
 * X = floor(log2(amax)) - 2 (2 = emax of E2M1), clamped to [-127, 127]
 * (amax = 0 gives -127); scale[m, b] = X + 127 (E8M0); elements
 * E2M1(x * 2^-X) (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), round to nearest
 * even, saturating to +-6, sign kept.  q: uint8 [M, K/2] row-major, two
 * codes a byte, element 2j in the low nibble (4-byte aligned); scale: uint8
 * [M, K/32] row-major.  x: bf16 [M, ldx].  K % 32 == 0.  Any M >= 1.
 */
int mr_mxfp4_quant(const void *x, int64_t ldx, int M, int K, uint8_t *q,
                   uint8_t *scale, void *stream);

/*
 * Every option of the one-launch route (a6) in one call.  Fields as the
 * arguments of mr_moe_route_sort_quant and mr_moe_route_sort_quant_norm;
 * in addition:
 *  - rstd == NULL: x is the router input as given; else x holds the
 *    un-normalised residual rows and the route runs on the norm's scale
 *    (rstd, norm_weight, norm_kind as in mr_moe_route_sort_quant_norm);
 *  - quant_format: MR_QUANT_NONE (q and scale ignored), MR_QUANT_MXFP8
 *    (q [M, K]) or MR_QUANT_MXFP4 (q [M, K/2], as mr_mxfp4_quant); q must be
 *    8-byte aligned.  An unknown format returns MR_ERR_INVALID_ARG.
 *  - shared_w13 != NULL: the shared expert's gate/up projection and SwiGLU
 *    run in the same launch, on extra clusters beside the route's (sglang
 *    #46691 Summary: the router fused with the shared expert's fp8 SwiGLU,
 *    the one-launch decode router running the shared expert's gate_up),
 *    writing shared_act exactly as mr_shared_gate_up (on the norm's scale
 *    too when rstd != NULL: the shared expert reads the norm's output).
 *    M <= 16, else MR_ERR_UNSUPPORTED.
 * Every output is bitwise equal to the unfused calls on the same input
 * (mr_norm_apply first when rstd != NULL; mr_mxfp8_quant or mr_mxfp4_quant
 * for the quant; mr_shared_gate_up for the shared expert).  The caller owns
 * the struct; it is read during the call only.  (ABI version 2 appended the
 * shared_* fields.)
 */
typedef struct mr_route_params {
    const void *x;               /* bf16 [M, ldx] */
    int64_t ldx;
    const float *rstd;           /* NULL, or fp32 [M] */
    const void *norm_weight;     /* bf16 [K] (with rstd) */
    int norm_kind;               /* MR_NORM_* (with rstd) */
    const void *w;               /* bf16 [N, K] gate weight */
    int M, N, K, topk, scoring;
    const float *sel_bias;       /* fp32 [N] or NULL (sigmoid scoring) */
    int renormalize;
    int block;
    int quant_format;            /* MR_QUANT_* */
    float *logits;               /* fp32 [M, N] */
    int32_t *topk_ids;           /* [M, topk] */
    float *topk_weights;         /* [M, topk] */
    int32_t *sorted_token_ids;   /* [capacity] */
    int32_t *expert_ids;         /* [capacity / block] */
    int32_t *num_tokens_post_padded;  /* [1] */
    int64_t capacity;
    uint8_t *q;
    uint8_t *scale;              /* uint8 [M, K/32] */
    void *scratch;
    size_t scratch_bytes;
    /* the shared expert's gate/up projection + SwiGLU in the same launch
     * (shared_w13 == NULL: none); see mr_shared_gate_up.  M <= 16. */
    const uint8_t *shared_w13;        /* E4M3 [2 * shared_inter, K] */
    const uint8_t *shared_w13_scale;  /* E8M0 [2 * shared_inter, K / 32] */
    int shared_inter;                 /* I */
    void *shared_act;                 /* bf16 [M, shared_inter] */
} mr_route_params;

int mr_moe_route(const mr_route_params *params, void *stream);

/*
 * a6 on the norm's scale [sgl-amd-mono #56 page, entry #59 "[Perf]
 * minimax_m31: Run o_proj in the launch, route on the norm's scale, read B
 * operands from LDS", Modifications, "Route on the norm's scale": the
 * RMSNorm in front of the router publishes each token's rstd, and the router
 * normalises its own columns of the residual sum instead of waiting for the
 * norm's output].  The router input is
 *     xn[m, k] = bf16( (sres[m, k] * rstd[m]) * s[k] ),
 * both products fp32 with round-to-nearest-even, the bf16 store rounding to
 * nearest even; s = norm_weight[k] (MR_NORM_RMS) or 1 + norm_weight[k] in
 * fp32 (MR_NORM_GEMMA, the Gemma RMSNorm of the MiniMax-M3 producers in
 * sglang #46691, "Changes to existing kernels").  Every output (logits, ids,
 * weights, sort, and q / scale, the MXFP8 of xn) is bitwise equal to
 * mr_norm_apply -> mr_moe_route_sort_quant on the same inputs.
 * sres: bf16 [M, ldx] (the un-normalised residual rows, 16-byte aligned);
 * rstd: fp32 [M] (4-byte aligned), read after the previous kernel on the
 * stream has finished; norm_weight: bf16 [K] (16-byte aligned).  The rest as
 * mr_moe_route_sort_quant, with its limits.  A NULL rstd or norm_weight, or
 * an unknown norm_kind, returns MR_ERR_INVALID_ARG.
 */
int mr_moe_route_sort_quant_norm(const void *sres, int64_t ldx, const float *rstd,
                                 const void *norm_weight, int norm_kind, const void *w,
                                 int M, int N, int K, int topk, int scoring,
                                 const float *sel_bias, int renormalize, int block,
                                 float *logits, int32_t *topk_ids, float *topk_weights,
                                 int32_t *sorted_token_ids, int32_t *expert_ids,
                                 int32_t *num_tokens_post_padded, int64_t capacity,
                                 uint8_t *q, uint8_t *scale,
                                 void *scratch, size_t scratch_bytes, void *stream);

/*
 * The router input on the norm's scale, written out (the norm's XN; the
 * unfused half of mr_moe_route_sort_quant_norm): xn[m, k] as defined there,
 * row-major [M, K], 16-byte aligned.  Any M >= 1; K % 8 == 0 (else
 * MR_ERR_UNSUPPORTED).  One launch.
 */
int mr_norm_apply(const void *sres, int64_t ldx, const float *rstd, const void *norm_weight,
                  int norm_kind, int M, int K, void *xn, void *stream);

/*
 * The shared expert's gate/up projection and SwiGLU [sglang #46691 Summary:
 * the router GEMV fused with the shared expert's fp8 SwiGLU, the MiniMax-M3.1
 * shared expert's 1536 x 6144 gate_up; sgl-amd-mono #56 page, Modifications:
 * the shared expert on its MXFP8 values with bf16 activations]:
 *   W[r, k]   = E4M3(w13[r, k]) * 2^(w13_scale[r, k / 32] - 127)
 *   h[m, r]   = sum_k x[m, k] W[r, k]          (fp32 accumulation)
 *   act[m, i] = silu(h[m, i]) * h[m, I + i],   silu(v) = v / (1 + e^-v)
 * rounded to bf16 (nearest even).  x: bf16 [M, ldx]; w13: E4M3 codes
 * [2I, K] row-major, rows [0, I) the gate projection and [I, 2I) the up
 * projection (16-byte aligned); w13_scale: E8M0 bytes [2I, K / 32] (below
 * 255, NaN); act: bf16 [M, I] (4-byte aligned).  Each 32-wide block of a
 * row is summed in fp32 (products exact) and scaled by its factor with one
 * fused multiply-add; the K range is split over the CTAs of a cluster as in
 * the router GEMV and the partial sums are added in a fixed order, so the
 * result is deterministic.  Each CTA stages its K slice of the weights in
 * shared memory (bulk async copies, issued before it waits on the previous
 * kernel); the number of clusters is the most that run beside the route's
 * at once.  A CTA whose slice of x converts to f16 exactly (zero, or
 * 2^-17 <= |x| < 2^16) runs f16 MMAs on the codes converted to f16, else
 * bf16 MMAs: the products are exact either way.
 * The output keeps finite values when the
 * weights' scale bytes are at most 246 (|W| below 2^128).  1 <= M <= 16,
 * K % 512 == 0, I % 8 == 0, and I up to 1536 at K = 6144 (at most 48 row
 * tiles x k-parts per CTA over at most 16 clusters), else
 * MR_ERR_UNSUPPORTED.  One launch.  In mr_moe_route (mr_route_params.shared_w13) the same work
 * joins the routing launch.
 */
int mr_shared_gate_up(const void *x, int64_t ldx, const uint8_t *w13, const uint8_t *w13_scale, int M, int K,
                      int I, void *act, void *stream);

/* Bytes of the library-owned scratch of mr_router_gemv_noalloc (8 MiB). */
#define MR_NOALLOC_SCRATCH_BYTES 8388608

/*
 * Router GEMV that allocates nothing and takes no scratch argument.  The
 * pages have no counterpart: this entry point exists for callers that cannot
 * call cudaMalloc or cannot hand this library a scratch buffer -- plugins
 * whose host framework owns all device memory and exposes no allocator to
 * them, or code paths that must not enter the driver's allocator (it can
 * synchronise the device and can fail once memory is fragmented).
 * Same arithmetic as mr_router_gemv's split-K kernel with the last-arriver
 * fixup (for every M here, including M <= 64, where mr_router_gemv runs its
 * cluster kernel instead, so the two agree within fp32 rounding, not bit
 * for bit).  The scratch is MR_NOALLOC_SCRATCH_BYTES of device memory that
 * this library declares at file scope; every GPU that loads the library
 * holds it until the process exits.
 *  - Every call looks up the array's device address on the current device
 *    (host code cannot use the array's name as an address).  The FIRST call
 *    in a device's context -- including the first after that context was
 *    destroyed and created again, e.g. by cudaDeviceReset, which reloads the
 *    library's device code -- zeroes the array's counters with one
 *    cudaMemsetAsync on the call's stream before its launch; make that first
 *    call before any stream capture.
 *  - With MR_LAUNCH_CHECK_SCRATCH set, each call verifies that the array's
 *    counters are zero before it launches (see mr_set_launch_flags).
 *  - Every call on a device shares the one array, and the array keeps the
 *    last call's contents: calls that can overlap on the GPU (different
 *    streams, concurrent threads) race and corrupt each other's results.
 *    Issue them on one stream, or serialise them.
 *  - Problems whose split-K partials do not fit (32 KiB counters plus
 *    SPLIT_K*M*N*4 bytes; e.g. M = 512, N = 128, K = 6144 fits) return
 *    MR_ERR_UNSUPPORTED without launching; so do shapes outside
 *    mr_router_gemv's cover.  Arguments as mr_router_gemv.
 */
int mr_router_gemv_noalloc(const void *x, int64_t ldx, const void *w, float *logits,
                           int M, int N, int K, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ROUTE_H */
