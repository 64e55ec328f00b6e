// Gate (a3), sort (a4) and MXFP8 quant (a5) launches.
#include "internal.h"
#include "sort.cuh"
#include "topk.cuh"

namespace mr {

// ------------------------------------------------------------------ gate

constexpr int kTopkWarps = 4;

template <int NPL, bool SIG>
__global__ void __launch_bounds__(32 * kTopkWarps) topk_kernel(TopkArgs a) {
    pdl_trigger();
    pdl_wait();
    const int m = blockIdx.x * kTopkWarps + (threadIdx.x >> 5);
    if (m < a.M) warp_topk_row<NPL, SIG>(a, m, nullptr);
}

int topk_npl(int N) { return N <= 128 ? 4 : N <= 256 ? 8 : N <= 512 ? 16 : 32; }

cudaError_t launch_topk(const float* logits, int M, int N, int topk, int scoring,
                        const float* bias, int renormalize, int32_t* ids, float* weights,
                        cudaStream_t st) {
    TopkArgs a{logits, bias, ids, weights, M, N, topk, scoring, renormalize,
               (launch_flags() & 8) ? 1 : 0};
    dim3 grid((M + kTopkWarps - 1) / kTopkWarps);
    const dim3 block(32 * kTopkWarps);
    const bool sig = scoring == 1;
    switch (topk_npl(N)) {
        case 4: return sig ? launch_kernel(topk_kernel<4, true>, grid, block, 0, st, a)
                           : launch_kernel(topk_kernel<4, false>, grid, block, 0, st, a);
        case 8: return sig ? launch_kernel(topk_kernel<8, true>, grid, block, 0, st, a)
                           : launch_kernel(topk_kernel<8, false>, grid, block, 0, st, a);
        case 16: return sig ? launch_kernel(topk_kernel<16, true>, grid, block, 0, st, a)
                            : launch_kernel(topk_kernel<16, false>, grid, block, 0, st, a);
        default: return sig ? launch_kernel(topk_kernel<32, true>, grid, block, 0, st, a)
                            : launch_kernel(topk_kernel<32, false>, grid, block, 0, st, a);
    }
}

// ------------------------------------------------------------------ sort

cudaError_t ensure_smem(const void* func, int bytes, int* done_per_device) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (__atomic_load_n(&done_per_device[dev], __ATOMIC_ACQUIRE) >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
    if (e == cudaSuccess) __atomic_store_n(&done_per_device[dev], 160 * 1024, __ATOMIC_RELEASE);
    return e;
}

struct SortWork {
    int* chunk_cnt;   // [C][N]
    int* chunk_off;   // [C][N]
    int* lrank;       // [n_assign]
    int* start;       // [N] padded start of each expert's run
    int* cnt;         // [N] assignments per expert
    int* total;       // [1]
};

__host__ __device__ inline SortWork sort_work(void* scratch, int n_assign, int N) {
    const int C = (n_assign + kSortChunk - 1) / kSortChunk;
    int* base = reinterpret_cast<int*>(static_cast<char*>(scratch) + kWorkOffset);
    SortWork w;
    w.chunk_cnt = base;
    w.chunk_off = w.chunk_cnt + (size_t)C * N;
    w.lrank = w.chunk_off + (size_t)C * N;
    w.start = w.lrank + n_assign;
    w.cnt = w.start + N;
    w.total = w.cnt + N;
    return w;
}

size_t sort_work_bytes(int n_assign, int N) {
    const size_t C = (n_assign + kSortChunk - 1) / kSortChunk;
    return sizeof(int) * (2 * C * N + (size_t)n_assign + 2 * (size_t)N + 4);
}

// Pass 1 of the multi-CTA sort: per-chunk counts and chunk-local stable
// ranks; the last chunk to finish turns the counts into chunk offsets and
// the padded expert starts.
__global__ void __launch_bounds__(kSortThreads) sort_count_kernel(SortArgs a, SortWork w,
                                                                  unsigned* counter) {
    extern __shared__ __align__(16) int sm[];
    __shared__ unsigned s_ticket;
    pdl_trigger();
    pdl_wait();
    const int nw = blockDim.x >> 5, tid = threadIdx.x, nthr = blockDim.x;
    const int C = gridDim.x, c = blockIdx.x, N = a.N;
    const int beg = c * kSortChunk, n = min(kSortChunk, a.n_assign - beg);
    RankSmem rs{sm, sm + nw * N, sm + nw * N + N};
    const int* ids = stage_ids(a.ids + beg, n, rs.lrank + kSortChunk);
    const int seg = cta_rank(ids, n, N, rs);
    for (int i = tid; i < n; i += nthr) {
        const int e = ids[i];
        if (e >= 0 && e < N) w.lrank[beg + i] = rs.wcnt[(i / seg) * N + e] + rs.lrank[i];
    }
    for (int e = tid; e < N; e += nthr) w.chunk_cnt[(size_t)c * N + e] = rs.cnt[e];
    const unsigned t = cta_ticket(counter, &s_ticket);
    if (t != (unsigned)(C - 1)) return;
    int* start = rs.lrank;  // reuse
    int* warp_tot = start + N;
    const int B = a.block;
    for (int e = tid; e < N; e += nthr) {
        int run = 0;
        for (int c0 = 0; c0 < C; c0 += kLoadBatch) {  // chunk counts kLoadBatch at a time
            int v[kLoadBatch];
#pragma unroll
            for (int u = 0; u < kLoadBatch; ++u)
                v[u] = c0 + u < C ? __ldcg(w.chunk_cnt + (size_t)(c0 + u) * N + e) : 0;
#pragma unroll
            for (int u = 0; u < kLoadBatch; ++u) {
                if (c0 + u < C) w.chunk_off[(size_t)(c0 + u) * N + e] = run;
                run += v[u];
            }
        }
        rs.cnt[e] = run;
        start[e] = (run + B - 1) / B * B;
    }
    __syncthreads();
    const int total = block_exclusive_scan(start, N, warp_tot);
    for (int e = tid; e < N; e += nthr) {
        w.start[e] = start[e];
        w.cnt[e] = rs.cnt[e];
    }
    // expert_ids of the real blocks, written here while the counts are at hand
    for (int e = tid; e < N; e += nthr) {
        const int st = start[e], p = (rs.cnt[e] + B - 1) / B * B;
        for (int b = st / B; b < (st + p) / B; ++b) a.expert_ids[b] = e;
    }
    if (tid == 0) {
        *w.total = total;
        *a.ntpp = total;
        *counter = 0u;
    }
}

// Pass 2: place every assignment, fill the padding and the tail.
__global__ void __launch_bounds__(kSortThreads) sort_scatter_kernel(SortArgs a, SortWork w) {
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x, nthr = blockDim.x, c = blockIdx.x, N = a.N, B = a.block;
    const int beg = c * kSortChunk, n = min(kSortChunk, a.n_assign - beg);
    for (int base = tid; base < n; base += nthr * kLoadBatch) {  // two dependent rounds per batch
        int e[kLoadBatch], lr[kLoadBatch], pos[kLoadBatch];
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {
            const int i = base + u * nthr;
            e[u] = i < n ? a.ids[beg + i] : -1;
            lr[u] = i < n ? w.lrank[beg + i] : 0;
        }
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {
            const bool ok = e[u] >= 0 && e[u] < N;
            pos[u] = ok ? w.start[e[u]] + w.chunk_off[(size_t)c * N + e[u]] + lr[u] : -1;
        }
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u)
            if (pos[u] >= 0) a.sorted[pos[u]] = beg + base + u * nthr;
    }
    const int64_t gt = (int64_t)c * nthr + tid, T = (int64_t)gridDim.x * nthr;
    const int total = *w.total, sentinel = a.n_assign;
    for (int64_t e = gt; e < N; e += T) {
        const int cnt = w.cnt[e];
        const int st = w.start[e], p = (cnt + B - 1) / B * B;
        for (int i = cnt; i < p; ++i) a.sorted[st + i] = sentinel;
    }
    for (int64_t i = total + gt; i < a.capacity; i += T) a.sorted[i] = sentinel;
    for (int64_t b = total / B + gt; b < a.capacity / B; b += T) a.expert_ids[b] = -1;
}

static int g_sort_count_smem[64];

cudaError_t launch_sort(const int32_t* ids, int M, int topk, int N, int block, int32_t* sorted,
                        int32_t* expert_ids, int32_t* ntpp, int64_t capacity, void* scratch,
                        cudaStream_t st) {
    SortArgs a{ids, M * topk, N, block, sorted, expert_ids, ntpp, capacity};
    if (a.n_assign <= kPSortMaxAssign)
        return launch_psort(a, M, topk, nullptr, 0, 0, nullptr, nullptr, 0, false, st);
    const int nw = kSortThreads / 32;
    const int C = (a.n_assign + kSortChunk - 1) / kSortChunk;
    SortWork w = sort_work(scratch, a.n_assign, N);
    const int smem = 4 * (nw * N + N + 2 * kSortChunk);
    cudaError_t e = ensure_smem((const void*)sort_count_kernel, smem, g_sort_count_smem);
    if (e != cudaSuccess) return e;
    unsigned* counter = static_cast<unsigned*>(scratch) + kSortCounterSlot;
    e = launch_kernel(sort_count_kernel, dim3(C), dim3(kSortThreads), smem, st, a, w, counter);
    if (e != cudaSuccess) return e;
    return launch_kernel(sort_scatter_kernel, dim3(C), dim3(kSortThreads), 0, st, a, w);
}

// ------------------------------------------------------------------ quant

// One lane quantises 8 consecutive elements; a lane quad is one 32-block.
// Work is cut into tiles of one row x 32 * kQuantUnroll 16-byte vectors (a
// warp per tile, kQuantUnroll loads in flight per lane): one 32-bit division
// per tile locates it, so the per-element cost stays the quantiser's own.
constexpr int kQuantThreads = 256;
constexpr int kQuantUnroll = 4;
constexpr int kQuantTileVec = 32 * kQuantUnroll;
constexpr int kSortQuantThreads = 512;

// Tiles warp_id, warp_id + nwarps, ... of the quantisation of x [M, K]
// (the whole warp takes part).  FP4: MXFP4 (E2M1 codes, two a byte,
// q [M, K/2]); else MXFP8 (E4M3, q [M, K]).
template <bool FP4>
__device__ __forceinline__ void quant_tiles(const uint16_t* x, int64_t ldx, int M, int K, uint8_t* q,
                                            uint8_t* scale, int warp_id, int nwarps) {
    const int lane = threadIdx.x & 31;
    const int vpr = K / 8;                                   // vectors per row
    const int tpr = (vpr + kQuantTileVec - 1) / kQuantTileVec;  // tiles per row
    const int K32 = K / 32;
    // tile t = (row r, chunk ch) with t = r * tpr + ch; the stride nwarps
    // advances (r, ch) by (dq, dr) with a carry: no division per tile
    const int dq = nwarps / tpr, dr = nwarps - dq * tpr;
    int r = warp_id / tpr, ch = warp_id - r * tpr;
    for (; r < M; r += dq, ch += dr) {
        if (ch >= tpr) {
            ch -= tpr;
            ++r;
            if (r >= M) break;
        }
        const int c0 = ch * kQuantTileVec + lane;
        const uint16_t* xr = x + (int64_t)r * ldx;
        uint4 v[kQuantUnroll];
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const int c = c0 + u * 32;
            v[u] = c < vpr ? ld_stream_v4(xr + c * 8) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const int c = c0 + u * 32;
            unsigned sb;
            if constexpr (FP4) {
                const uint32_t q4 = mx4_quant_quad(v[u], &sb);
                if (c < vpr) *reinterpret_cast<uint32_t*>(q + (int64_t)r * (K / 2) + c * 4) = q4;
            } else {
                const uint2 q8 = mx_quant_quad(v[u], &sb);
                if (c < vpr) *reinterpret_cast<uint2*>(q + (int64_t)r * K + c * 8) = q8;
            }
            if (c < vpr && (lane & 3) == 0) scale[(int64_t)r * K32 + c / 4] = (uint8_t)sb;
        }
    }
}

template <bool FP4>
__global__ void __launch_bounds__(kQuantThreads) mx_quant_kernel(const uint16_t* x, int64_t ldx, int M, int K,
                                                                 uint8_t* q, uint8_t* scale) {
    pdl_trigger();
    pdl_wait();
    quant_tiles<FP4>(x, ldx, M, K, q, scale, (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5),
                     (int)((gridDim.x * blockDim.x) >> 5));
}

// ------------------------------------------------------------------ parallel sort (+ quant)
//
// The sort of up to kPSortMaxAssign assignments in ONE launch over many CTAs
// with no hand-off between them: every CTA counts the assignments of every
// expert (all ids, read through L2) and those of the rows before its own
// block, so it knows the padded start of each expert and the final position
// of each of its own assignments without waiting for another CTA.  CTA c
// places the assignments of its token rows [c R, (c + 1) R), writes the
// padding and the block ids of experts c, c + G, ..., its share of the tail
// and of num_tokens_post_padded, and (with a format) the MX quantisation of
// its rows: in token order, or at the sorted positions of the rows'
// assignments (the zero rows of the padding by the CTA of their expert).

// hist[e] += number of ids[beg, end) equal to e (ids outside [0, N) are
// skipped).  Each warp counts into its own row of warp_hist ([warps][N],
// zero on entry and on return) with shared atomics, kLoadBatch coalesced
// loads in flight per thread; the rows are then added into hist.  (Warp-wide
// peer matching per 32 ids ran on a low-throughput pipe and made the count
// the long pole of the sort.)
__device__ __forceinline__ void psort_hist(const int32_t* ids, int beg, int end, int N, int* warp_hist, int* hist) {
    const int tid = threadIdx.x, nthr = blockDim.x, nw = nthr >> 5;
    int* my = warp_hist + (tid >> 5) * N;
    for (int base = beg + tid; base < end; base += nthr * kLoadBatch) {
        int e[kLoadBatch];
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {
            const int i = base + u * nthr;
            e[u] = i < end ? ids[i] : -1;
        }
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u)
            if (e[u] >= 0 && e[u] < N) atomicAdd(&my[e[u]], 1);
    }
    __syncthreads();
    for (int e = tid; e < N; e += nthr) {
        int sum = 0;
        for (int w = 0; w < nw; ++w) {
            sum += warp_hist[w * N + e];
            warp_hist[w * N + e] = 0;
        }
        hist[e] += sum;
    }
    __syncthreads();
}

// MX quantisation of rows x[0, rows) written to the sorted positions of their
// assignments: pos[r * k + j] (or -1: not placed).  The same tile walk and
// arithmetic as quant_tiles; each tile's codes and scales go to k rows.
template <bool FP4>
__device__ __forceinline__ void quant_rows_to_positions(const uint16_t* x, int64_t ldx, int rows, int K,
                                                        const int* pos, int k, uint8_t* q, uint8_t* scale,
                                                        int warp_id, int nwarps) {
    const int lane = threadIdx.x & 31;
    const int vpr = K / 8, tpr = (vpr + kQuantTileVec - 1) / kQuantTileVec, K32 = K / 32;
    const int64_t qk = FP4 ? K / 2 : K;
    for (int t = warp_id; t < rows * tpr; t += nwarps) {
        const int r = t / tpr, c0 = (t - r * tpr) * kQuantTileVec + lane;
        const uint16_t* xr = x + (int64_t)r * ldx;
        uint4 v[kQuantUnroll];
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const int c = c0 + u * 32;
            v[u] = c < vpr ? ld_ro_v4(xr + c * 8) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const int c = c0 + u * 32;
            unsigned sb;
            uint2 q8 = make_uint2(0u, 0u);
            uint32_t q4 = 0u;
            if constexpr (FP4)
                q4 = mx4_quant_quad(v[u], &sb);
            else
                q8 = mx_quant_quad(v[u], &sb);
            if (c >= vpr) continue;
            for (int j = 0; j < k; ++j) {
                const int p = pos[r * k + j];
                if (p < 0) continue;
                if constexpr (FP4)
                    *reinterpret_cast<uint32_t*>(q + (int64_t)p * qk + c * 4) = q4;
                else
                    *reinterpret_cast<uint2*>(q + (int64_t)p * qk + c * 8) = q8;
                if ((lane & 3) == 0) scale[(int64_t)p * K32 + c / 4] = (uint8_t)sb;
            }
        }
    }
}

struct PSortArgs {
    SortArgs s;
    int M, k, rows_per;   // token rows per CTA
    int staged;           // 1: every id staged in shared memory (n_assign <= kPSortStageMax)
    const uint16_t* x;    // stage-1 activations [M, ldx] (FMT != 0)
    int64_t ldx;
    int K;
    uint8_t* q;           // [M or capacity rows, K or K/2]
    uint8_t* scale;       // [M or capacity rows, K/32]
};

// Shared-memory ints of one CTA: pre, tot, start [N] each, 32 scan slots, own
// ids and positions [own], the ranking tables (warps x N, N, own).
__host__ __device__ constexpr int psort_smem_ints(int nwarps, int N, int own) {
    return 3 * N + 32 + 2 * own + nwarps * N + N + own;
}

// FMT: 0 sort only, 1 MXFP8, 2 MXFP4; SORTED: quantised rows at the sorted
// positions (q, scale with capacity rows) instead of token order.
template <int FMT, bool SORTED>
__global__ void __launch_bounds__(kSortQuantThreads) psort_kernel(PSortArgs a) {
    extern __shared__ __align__(16) int sm[];
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x, nthr = blockDim.x, nw = nthr >> 5, warp = tid >> 5;
    const int N = a.s.N, B = a.s.block, k = a.k, G = (int)gridDim.x, c = (int)blockIdx.x;
    const int n_all = a.s.n_assign, sentinel = n_all;
    const int m0 = min(c * a.rows_per, a.M), m1 = min(m0 + a.rows_per, a.M);
    const int f0 = m0 * k, n_own = (m1 - m0) * k, own_max = a.rows_per * k;
    int* pre = sm;                   // assignments per expert in rows [0, m0)
    int* tot = pre + N;              // assignments per expert, all rows
    int* start = tot + N;            // padded start of each expert's run
    int* warp_tot = start + N;       // scan slots
    int* own_ids = warp_tot + 32;    // this CTA's ids
    int* own_pos = own_ids + own_max;  // their sorted positions (-1: not placed)
    RankSmem rs{own_pos + own_max, own_pos + own_max + nw * N, own_pos + own_max + nw * N + N};
    for (int e = tid; e < N; e += nthr) {
        pre[e] = 0;
        tot[e] = 0;
    }
    for (int i = tid; i < nw * N; i += nthr) rs.wcnt[i] = 0;  // the per-warp counts of psort_hist
    // up to kPSortStageMax ids: all of them to shared memory in one round of
    // loads, counted from there (and this CTA's own ids are a slice of them)
    const int32_t* ids = a.s.ids;
    if (a.staged) {
        int* all = own_pos + own_max + nw * N + N + own_max;
        stage_ids(a.s.ids, n_all, all);
        ids = all;
        for (int i = tid; i < n_own; i += nthr) own_ids[i] = all[f0 + i];
    } else {
        for (int i = tid; i < n_own; i += nthr) own_ids[i] = __ldg(a.s.ids + f0 + i);
    }
    __syncthreads();
    psort_hist(ids, 0, f0, N, rs.wcnt, pre);
    psort_hist(ids, f0, n_all, N, rs.wcnt, tot);
    for (int e = tid; e < N; e += nthr) {
        const int t = tot[e] + pre[e];
        tot[e] = t;
        start[e] = (t + B - 1) / B * B;
    }
    __syncthreads();
    const int total = block_exclusive_scan(start, N, warp_tot);
    // stable ranks inside this CTA's block, offset by the rows before it
    const int seg = cta_rank(own_ids, n_own, N, rs);
    for (int i = tid; i < n_own; i += nthr) {
        const int e = own_ids[i];
        int p = -1;
        if (e >= 0 && e < N) {
            p = start[e] + pre[e] + rs.wcnt[(i / seg) * N + e] + rs.lrank[i];
            a.s.sorted[p] = f0 + i;
        }
        own_pos[i] = p;
    }
    // padding and block ids of experts c, c + G, ... (a thread per expert);
    // the tail past the total
    for (int e = c + G * tid; e < N; e += G * nthr) {
        const int st = start[e], t = tot[e], pd = (t + B - 1) / B * B;
        for (int i = t; i < pd; ++i) a.s.sorted[st + i] = sentinel;
        for (int b = st / B; b < (st + pd) / B; ++b) a.s.expert_ids[b] = e;
    }
    {
        const int64_t gt = (int64_t)c * nthr + tid, T = (int64_t)G * nthr;
        for (int64_t i = total + gt; i < a.s.capacity; i += T) a.s.sorted[i] = sentinel;
        for (int64_t b = total / B + gt; b < a.s.capacity / B; b += T) a.s.expert_ids[b] = -1;
    }
    if (c == 0 && tid == 0) *a.s.ntpp = total;
    if constexpr (FMT != 0) {
        constexpr bool FP4 = FMT == 2;
        const int K = a.K;
        const int64_t qk = FP4 ? K / 2 : K, K32 = K / 32;
        if constexpr (!SORTED) {
            quant_tiles<FP4>(a.x + (int64_t)m0 * a.ldx, a.ldx, m1 - m0, K, a.q + (int64_t)m0 * qk,
                             a.scale + (int64_t)m0 * K32, warp, nw);
        } else {
            __syncthreads();  // own_pos complete
            quant_rows_to_positions<FP4>(a.x + (int64_t)m0 * a.ldx, a.ldx, m1 - m0, K, own_pos, k, a.q, a.scale,
                                         warp, nw);
            // zero rows at the padding positions of experts c, c + G, ...
            for (int e = c; e < N; e += G) {
                const int st = start[e], t = tot[e], pd = (t + B - 1) / B * B;
                const int64_t nq = (int64_t)(pd - t) * (qk / 8);  // 8-byte words (qk % 16 == 0)
                uint2* qz = reinterpret_cast<uint2*>(a.q + (int64_t)(st + t) * qk);
                for (int64_t i = tid; i < nq; i += nthr) qz[i] = make_uint2(0u, 0u);
                const int64_t ns = (int64_t)(pd - t) * K32;
                uint8_t* sz = a.scale + (int64_t)(st + t) * K32;
                for (int64_t i = tid; i < ns; i += nthr) sz[i] = 0;
            }
        }
    }
}

static int g_psort_smem[6][64];

cudaError_t launch_psort(const SortArgs& s, int M, int topk, const void* x, int64_t ldx, int K, uint8_t* q,
                         uint8_t* scale, int fmt, bool sorted_rows, cudaStream_t st) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    // rows per CTA: at most one CTA per SM (each counts every id), and at
    // most kPSortMaxOwn assignments placed by one CTA
    int rows_per = (M + sms - 1) / sms;
    if (rows_per * topk > kPSortMaxOwn) rows_per = kPSortMaxOwn / topk;
    if (rows_per < 1) rows_per = 1;
    const int G = (M + rows_per - 1) / rows_per;
    const int staged = s.n_assign <= kPSortStageMax ? 1 : 0;
    PSortArgs a{s, M, topk, rows_per, staged, static_cast<const uint16_t*>(x), ldx, K, q, scale};
    const int nw = kSortQuantThreads / 32;
    const int smem = 4 * (psort_smem_ints(nw, s.N, rows_per * topk) + (staged ? s.n_assign : 0));
    void (*kernel)(PSortArgs) = nullptr;
    int slot = 0;
    if (fmt == 0) {
        kernel = psort_kernel<0, false>;
    } else if (fmt == 1) {
        kernel = sorted_rows ? psort_kernel<1, true> : psort_kernel<1, false>;
        slot = sorted_rows ? 2 : 1;
    } else {
        kernel = sorted_rows ? psort_kernel<2, true> : psort_kernel<2, false>;
        slot = sorted_rows ? 4 : 3;
    }
    e = ensure_smem((const void*)kernel, smem, g_psort_smem[slot]);
    if (e != cudaSuccess) return e;
    return launch_kernel(kernel, dim3((unsigned)G), dim3(kSortQuantThreads), smem, st, a);
}

cudaError_t launch_quant(const void* x, int64_t ldx, int M, int K, uint8_t* q, uint8_t* scale, bool fp4,
                         cudaStream_t st) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (int64_t)M * ((K / 8 + kQuantTileVec - 1) / kQuantTileVec);
    if (tiles >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
    const int64_t warps_per_cta = kQuantThreads / 32;
    int64_t ctas = (tiles + warps_per_cta - 1) / warps_per_cta;
    const int64_t cap = (int64_t)sms * 8;  // 8 resident CTAs per SM, grid-stride beyond
    if (ctas > cap) ctas = cap;
    return launch_kernel(fp4 ? mx_quant_kernel<true> : mx_quant_kernel<false>, dim3((unsigned)ctas),
                         dim3(kQuantThreads), 0, st, static_cast<const uint16_t*>(x), ldx, M, K, q, scale);
}

// Router input on the norm's scale, written out: xn[m, k] = bf16((x[m, k] *
// rstd[m]) * s[k]) for the unfused chain (one thread per 16-byte chunk,
// grid-stride).  xn is row-major [M, K].
__global__ void __launch_bounds__(256) norm_apply_kernel(const uint16_t* x, int64_t ldx, const float* rstd,
                                                         const uint16_t* g, int gemma, int M, int K,
                                                         uint16_t* xn) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int vpr = K / 8;
    const int tpr = (vpr + kQuantTileVec - 1) / kQuantTileVec;
    const int tiles = M * tpr;
    const int warp_id = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int nwarps = (int)((gridDim.x * blockDim.x) >> 5);
    for (int tile = warp_id; tile < tiles; tile += nwarps) {
        const int r = tile / tpr, c0 = (tile - r * tpr) * kQuantTileVec + lane;
        const float rs = __ldg(rstd + r);
        uint4 v[kQuantUnroll], gv[kQuantUnroll];
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const int c = c0 + u * 32;
            v[u] = c < vpr ? ld_stream_v4(x + (int64_t)r * ldx + c * 8) : make_uint4(0u, 0u, 0u, 0u);
            gv[u] = c < vpr ? ld_ro_v4(g + c * 8) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const int c = c0 + u * 32;
            if (c < vpr) *reinterpret_cast<uint4*>(xn + (int64_t)r * K + c * 8) = norm_chunk(v[u], gv[u], rs, gemma != 0);
        }
    }
}

cudaError_t launch_norm_apply(const void* x, int64_t ldx, const float* rstd, const void* g, int gemma, int M,
                              int K, void* xn, cudaStream_t st) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (int64_t)M * ((K / 8 + kQuantTileVec - 1) / kQuantTileVec);
    if (tiles >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
    int64_t ctas = (tiles + 7) / 8;  // 8 warps per CTA, a tile each
    const int64_t cap = (int64_t)sms * 8;
    if (ctas > cap) ctas = cap;
    return launch_kernel(norm_apply_kernel, dim3((unsigned)ctas), dim3(256), 0, st, static_cast<const uint16_t*>(x),
                         ldx, rstd, static_cast<const uint16_t*>(g), gemma, M, K, static_cast<uint16_t*>(xn));
}

}  // namespace mr
