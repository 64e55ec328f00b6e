// Sort of the (token, slot) assignments into padded per-expert blocks.
//
// The pages name aiter's multi-phase sort (sglang #46691 Summary) and give
// its key rule in the Kimi-K3 sort kernel's review diff (sglang #46652): the
// stable rank of an assignment is the number of earlier (token, slot) pairs
// routed to the same expert.  The layout (experts ascending, flat index
// f = m*k + j ascending inside an expert, runs padded to the block with the
// sentinel M*k, tail filled with the sentinel and expert id -1) is the
// plainest reading of that sort's outputs sorted_token_ids / expert_ids /
// num_tokens_post_padded.
//
// GB300 design (one CTA per <= 2048 assignments): each warp ranks its own
// contiguous segment 32 assignments at a time with __match_any_sync (peers
// on the same expert) and a per-warp counter row in shared memory; one pass
// per expert turns the per-warp counts into exclusive offsets; a block scan
// gives the padded expert starts; then every thread places its assignments.
// No atomics decide an order, so the result is unique.
#pragma once

#include "common.cuh"

namespace mr {

// Exclusive scan of a[0..n) in shared memory by the whole CTA; returns the
// total.  warp_tot needs 32 ints.
__device__ __forceinline__ int block_exclusive_scan(int* a, int n, int* warp_tot) {
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5;
    const int nw = nthr >> 5;
    const int per = (n + nthr - 1) / nthr;
    const int beg = min(tid * per, n), end = min(beg + per, n);
    int local = 0;
    for (int i = beg; i < end; ++i) local += a[i];
    int v = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += u;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(kFull, w, o);
            if (lane >= o) w += u;
        }
        warp_tot[lane] = w;
    }
    __syncthreads();
    int run = v - local + (warp > 0 ? warp_tot[warp - 1] : 0);
    for (int i = beg; i < end; ++i) {
        const int c = a[i];
        a[i] = run;
        run += c;
    }
    const int total = warp_tot[nw - 1];
    __syncthreads();
    return total;
}

// Shared-memory tables of one CTA's ranking pass.
struct RankSmem {
    int* wcnt;    // [nwarps][N]: per-warp counts, then per-warp exclusive offsets
    int* cnt;     // [N] assignments per expert in this CTA
    int* lrank;   // [n_assign] rank of the assignment inside its warp's segment
};

// Stable ranks of assignments ids[0..n) (global or shared), expert ids in
// [0, N).  After the call: cnt[e] = count of e; wcnt[w][e] = assignments of e
// in warps before w; the CTA-local stable rank of assignment i with expert e
// handled by warp w = i / seg is wcnt[w][e] + lrank[i].  Returns seg.
__device__ __forceinline__ int cta_rank(const int* ids, int n, int N, const RankSmem& s) {
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5;
    const int nw = nthr >> 5;
    for (int i = tid; i < nw * N; i += nthr) s.wcnt[i] = 0;
    __syncthreads();
    int seg = (n + nw - 1) / nw;
    seg = (seg + 31) & ~31;
    const int sbeg = warp * seg, send = min(sbeg + seg, n);
    int* my = s.wcnt + warp * N;
    for (int base = sbeg; base < send; base += 32) {
        const int i = base + lane;
        const int e = (i < send) ? ids[i] : -1;
        const bool valid = e >= 0 && e < N;
        const unsigned peers = __match_any_sync(kFull, valid ? e : (int)(0x40000000u | (unsigned)lane));
        const int before = __popc(peers & ((1u << lane) - 1u));
        const int basecnt = valid ? my[e] : 0;
        if (i < send) s.lrank[i] = basecnt + before;
        __syncwarp();
        if (valid && before == 0) my[e] = basecnt + __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    for (int e = tid; e < N; e += nthr) {
        int run = 0;
        for (int w = 0; w < nw; ++w) {
            const int c = s.wcnt[w * N + e];
            s.wcnt[w * N + e] = run;
            run += c;
        }
        s.cnt[e] = run;
    }
    __syncthreads();
    return seg;
}

struct SortArgs {
    const int32_t* ids;        // [M*k] (global)
    int n_assign;              // M*k
    int N, block;
    int32_t* sorted;           // [capacity]
    int32_t* expert_ids;       // [capacity / block]
    int32_t* ntpp;             // [1]
    int64_t capacity;
};

// Whole sort by one CTA (n_assign <= 2048).  ids_src may be shared or global.
// start needs N + ... ints; warp_tot 32 ints.
__device__ __forceinline__ void cta_sort(const SortArgs& a, const int* ids_src, const RankSmem& s,
                                         int* start, int* warp_tot,
                                         unsigned long long* trace = nullptr) {
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int N = a.N, B = a.block;
    const int seg = cta_rank(ids_src, a.n_assign, N, s);
    MR_TRACE_STAMP(trace, 7);
    for (int e = tid; e < N; e += nthr) start[e] = (s.cnt[e] + B - 1) / B * B;
    __syncthreads();
    const int total = block_exclusive_scan(start, N, warp_tot);
    MR_TRACE_STAMP(trace, 8);
    const int sentinel = a.n_assign;
    for (int i = tid; i < a.n_assign; i += nthr) {
        const int e = ids_src[i];
        if (e < 0 || e >= N) continue;
        const int w = i / seg;
        a.sorted[start[e] + s.wcnt[w * N + e] + s.lrank[i]] = i;
    }
    MR_TRACE_STAMP(trace, 9);
    for (int e = tid; e < N; e += nthr) {
        const int st = start[e], c = s.cnt[e], p = (c + B - 1) / B * B;
        for (int i = c; i < p; ++i) a.sorted[st + i] = sentinel;
        for (int b = st / B; b < (st + p) / B; ++b) a.expert_ids[b] = e;
    }
    for (int64_t i = total + tid; i < a.capacity; i += nthr) a.sorted[i] = sentinel;
    for (int64_t b = total / B + tid; b < a.capacity / B; b += nthr) a.expert_ids[b] = -1;
    if (tid == 0) *a.ntpp = total;
}

// Shared-memory ints the single-CTA sort needs for nwarps warps (its tables,
// then a copy of the ids: the ranking loop walks them in dependent steps, so
// they are staged once with every load in flight instead of one L2 round
// trip per step).
__host__ __device__ constexpr int cta_sort_smem_ints(int nwarps, int N, int n_assign) {
    return nwarps * N + 2 * N + n_assign + 32 + n_assign;
}

// Loads issued in groups of kLoadBatch per thread before their uses, so
// that a loop over global memory pays one L2 round trip per group.
constexpr int kLoadBatch = 8;

// ids[0..n) -> shared memory by the whole CTA (then a barrier).
__device__ __forceinline__ const int* stage_ids(const int32_t* ids, int n, int* dst) {
    const int nthr = blockDim.x;
    for (int base = threadIdx.x; base < n; base += nthr * kLoadBatch) {
        int v[kLoadBatch];
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {
            const int i = base + u * nthr;
            v[u] = i < n ? __ldg(ids + i) : 0;
        }
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {
            const int i = base + u * nthr;
            if (i < n) dst[i] = v[u];
        }
    }
    __syncthreads();
    return dst;
}

}  // namespace mr
