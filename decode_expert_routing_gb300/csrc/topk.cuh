// Warp-per-token top-k gate.
//
// The gate (sglang #46691 Summary; sglang #46652 Modifications): per token,
// pick the k experts with the largest selection key and weight them.
//   softmax: key = logit; weights = softmax of the selected logits
//            (renormalised) or the full softmax probabilities.
//   sigmoid: s = sigmoid(logit) correctly rounded to fp32, key = s + bias;
//            weights = s of the selected, renormalised or not.  Approximate
//            fp32 keys find the k-th largest key; only experts within
//            kSigmoidKeyMargin of it are re-scored exactly, then selected.
// Ties go to the lower expert id.
//
// GB300 design: one warp per token.  Lane l holds the keys of experts
// l, l+32, l+64, ... as order-preserving 32-bit images, so the loads of a
// row are coalesced.  Each of the k rounds takes the warp maximum with one
// redux.sync (max) and breaks ties with a second (min over the candidate
// ids), then only the winning lane rescans its NPL keys.  Slot j lives in
// lane j, which then forms the weight; sums use a fixed butterfly, so the
// result is deterministic.
#pragma once

#include "common.cuh"

namespace mr {

struct TopkArgs {
    const float* logits;   // [M, N]
    const float* bias;     // [N] or nullptr (sigmoid only)
    int32_t* ids;          // [M, k]
    float* weights;        // [M, k]
    int M, N, k;
    int scoring;           // 0 softmax, 1 sigmoid
    int renormalize;
    int slow_sigmoid;      // test hook: every exact sigmoid through double-double
};

// k rounds of the warp's largest key (ties to the lower id): slot r's id and
// logit go to lane r (my_id, my_val); the winners' keys are cleared.  Returns
// the k-th largest key.
template <int NPL>
__device__ __forceinline__ unsigned warp_select(unsigned (&key)[NPL], const float (&val)[NPL], int k, int* my_id,
                                                float* my_val) {
    const int lane = threadIdx.x & 31;
    unsigned best = 0u;
    int bestj = 0;
#pragma unroll
    for (int j = 0; j < NPL; ++j)
        if (key[j] > best) { best = key[j]; bestj = j; }
    unsigned kmax = 0u;
    for (int r = 0; r < k; ++r) {
        kmax = __reduce_max_sync(kFull, best);
        const unsigned cand = (best == kmax) ? (unsigned)(lane + 32 * bestj) : 0xFFFFFFFFu;
        const unsigned win = __reduce_min_sync(kFull, cand);
        const int owner = (int)(win & 31u), wj = (int)(win >> 5);
        float wv = 0.0f;
        if (lane == owner) {
            best = 0u;
            bestj = 0;
#pragma unroll
            for (int j = 0; j < NPL; ++j) {
                if (j == wj) { wv = val[j]; key[j] = 0u; }
                if (key[j] > best) { best = key[j]; bestj = j; }
            }
        }
        wv = __shfl_sync(kFull, wv, owner);
        if (lane == r) { *my_id = (int)win; *my_val = wv; }
    }
    return kmax;
}

// Gate of one token (row m) by one warp.  If ids_smem != nullptr the chosen
// ids are also written there (slot order).  Reads the logits through L2 so
// that rows written by other CTAs of the same launch are seen.
// (The exact sigmoid score goes through sigmoid_exact_call: the candidate
// loop below is unrolled over a lane's NPL keys, and inlined it put NPL
// copies of the evaluation into the kernel, 324 KB of code at NPL = 32.)
// SIG: the sigmoid gate (scoring 1), else softmax; a separate
// instantiation, so the softmax gate carries none of the sigmoid's code.
template <int NPL, bool SIG>
__device__ __forceinline__ void warp_topk_row(const TopkArgs& a, int m, int* ids_smem) {
    const int lane = threadIdx.x & 31;
    const float* row = a.logits + (int64_t)m * a.N;
    float val[NPL];
    unsigned key[NPL];
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
        const int id = lane + 32 * j;
        val[j] = id < a.N ? __ldcg(row + id) : 0.0f;
    }
    // keys: the logit (softmax), else the approximate sigmoid + bias
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
        const int id = lane + 32 * j;
        unsigned kv = 0u;  // below every real key: never selected while real keys remain
        if (id < a.N) {
            float sel = val[j];
            if constexpr (SIG) sel = __fadd_rn(sigmoid_approx(val[j]), a.bias ? __ldg(a.bias + id) : 0.0f);
            kv = ordered_key(sel);
        }
        key[j] = kv;
    }
    int my_id = 0;
    float my_val = 0.0f;  // slot lane's logit, or for the sigmoid gate its exact score
    if constexpr (SIG) {
        // the k-th largest approximate key bounds the candidates; they are
        // re-scored exactly, the others drop out, and the selection runs again
        unsigned probe[NPL];
        float score[NPL];
#pragma unroll
        for (int j = 0; j < NPL; ++j) probe[j] = key[j];
        const unsigned floor_key = sigmoid_candidate_floor(warp_select<NPL>(probe, val, a.k, &my_id, &my_val));
#pragma unroll
        for (int j = 0; j < NPL; ++j) {
            const int id = lane + 32 * j;
            const bool cand = id < a.N && key[j] >= floor_key;
            score[j] = cand ? sigmoid_exact_call(val[j], a.slow_sigmoid != 0) : 0.0f;
            key[j] = cand ? ordered_key(__fadd_rn(score[j], a.bias ? __ldg(a.bias + id) : 0.0f)) : 0u;
        }
        warp_select<NPL>(key, score, a.k, &my_id, &my_val);
    } else {
        warp_select<NPL>(key, val, a.k, &my_id, &my_val);
    }

    // weights: lane r < k owns slot r
    const bool live = lane < a.k;
    float num = 0.0f, den;
    if constexpr (SIG) {
        num = live ? my_val : 0.0f;
        den = a.renormalize ? warp_sum_fixed(num) : 1.0f;
    } else {
        const float lmax = __shfl_sync(kFull, my_val, 0);  // slot 0 holds the largest logit
        num = live ? expf(__fadd_rn(my_val, -lmax)) : 0.0f;
        if (a.renormalize) {
            den = warp_sum_fixed(num);
        } else {
            float part = 0.0f;
#pragma unroll
            for (int j = 0; j < NPL; ++j)
                if (lane + 32 * j < a.N) part = __fadd_rn(part, expf(__fadd_rn(val[j], -lmax)));
            den = warp_sum_fixed(part);
        }
    }
    if (live) {
        a.ids[(int64_t)m * a.k + lane] = my_id;
        a.weights[(int64_t)m * a.k + lane] = (SIG && !a.renormalize) ? num : __fdiv_rn(num, den);
        if (ids_smem) ids_smem[m * a.k + lane] = my_id;
    }
}

template <int NPL, bool SIG>
__device__ __forceinline__ void cta_topk_rows(const TopkArgs& a, int row_begin, int row_end,
                                              int* ids_smem) {
    const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    for (int m = row_begin + warp; m < row_end; m += nwarps) warp_topk_row<NPL, SIG>(a, m, ids_smem);
}

}  // namespace mr
