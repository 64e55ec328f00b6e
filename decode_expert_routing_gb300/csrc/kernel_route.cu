// The decode route as one thread-block cluster: router GEMV, split-K
// reduction, top-k gate, sort and MXFP8 quant in ONE launch for M <= 64.
//
// The pages' one-launch decode router (sglang #46691 Summary: a router for
// 1-16 tokens bitwise equal to router GEMV, gate and sort; sort + stage-1
// quant in one launch) chains its stages through global memory.  On GB300 a
// global last-arriver ticket costs ~0.7 us and a cluster barrier ~0.2 us, so
// this kernel keeps every hand-off inside one cluster of CS CTAs (16 when the
// device allows it, else 8) and distributed shared memory:
//
//   1. CTA c owns the K slice [c*K/CS, (c+1)*K/CS) for ALL experts.  Warps
//      take (8-expert tile, k-part) units and run m16n8k16 bf16 MMAs with
//      fp32 accumulation; gate-weight fragments come straight from global
//      memory with 16-byte loads issued before the kernel waits on its
//      predecessor (programmatic dependent launch), x fragments from the
//      CTA's x slice in shared memory.  The CTA quantises its x slice (MXFP8).
//   2. Split-K reduction: every unit's partial tile goes, as 8-byte DSMEM
//      stores, to the CTA that owns the tile's token rows (token m belongs to
//      CTA m / TOK).  After one cluster barrier the owner sums the CS*WPT
//      partials of each logit in a fixed order and writes the logits.
//   3. Gate: the owner runs the top-k of its rows, one warp per 128-expert
//      segment, segments merged by one warp; the chosen ids also go to CTA 0.
//   4. After a second cluster barrier CTA 0 sorts the assignments: since the
//      k ids of a token are distinct, the stable rank of (m, j) inside expert
//      e is popc(mask_e & ((1 << m) - 1)) where mask_e is the bitmask of the
//      tokens that chose e.
//
// No spin-waits: all waits are hardware cluster/CTA barriers.  Nothing is
// left in scratch, so no counter needs re-zeroing.  The GEMV alone (mode 0)
// is what the standalone router GEMV runs for M <= 64, so the logits of the
// two are bitwise equal.
#include "common.cuh"
#include "internal.h"
#include "route_plan.h"
#include "sort.cuh"

namespace mr {

__device__ __forceinline__ unsigned cluster_rank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync_acq_rel() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint32_t map_rank(uint32_t local, unsigned rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_f2(uint32_t addr, float a, float b) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}
__device__ __forceinline__ void st_cluster_s32(uint32_t addr, int v) {
    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint4 lds128(const void* p) {
    return *reinterpret_cast<const uint4*>(p);
}

// Top-k of candidates held NPL per lane (key = order-preserving image, 0 =
// absent; ids unique).  After the call lane r < k holds the r-th best
// (id, val, key), ties to the lower id.
template <int NPL>
__device__ __forceinline__ void warp_select(unsigned (&key)[NPL], const int (&id)[NPL],
                                            const float (&val)[NPL], int k, int* out_id,
                                            float* out_val, unsigned* out_key) {
    const int lane = threadIdx.x & 31;
    unsigned best = 0u;
    int bid = 0x7FFFFFFF;
    float bval = 0.0f;
#pragma unroll
    for (int j = 0; j < NPL; ++j)
        if (key[j] > best || (key[j] == best && key[j] != 0u && id[j] < bid)) {
            best = key[j];
            bid = id[j];
            bval = val[j];
        }
    int my_id = 0;
    float my_val = 0.0f;
    unsigned my_key = 0u;
    for (int r = 0; r < k; ++r) {
        const unsigned kmax = __reduce_max_sync(kFull, best);
        const unsigned cand = (best == kmax && best != 0u) ? (unsigned)bid : 0xFFFFFFFFu;
        const unsigned win = __reduce_min_sync(kFull, cand);
        const bool mine = cand == win && best != 0u;
        const int owner = __ffs(__ballot_sync(kFull, mine)) - 1;
        const float wv = __shfl_sync(kFull, bval, owner < 0 ? 0 : owner);
        if (lane == r) {
            my_id = (int)win;
            my_val = wv;
            my_key = kmax;
        }
        if (mine) {
            best = 0u;
            bid = 0x7FFFFFFF;
#pragma unroll
            for (int j = 0; j < NPL; ++j) {
                if ((unsigned)id[j] == win) key[j] = 0u;
                if (key[j] > best || (key[j] == best && key[j] != 0u && id[j] < bid)) {
                    best = key[j];
                    bid = id[j];
                    bval = val[j];
                }
            }
        }
    }
    *out_id = my_id;
    *out_val = my_val;
    *out_key = my_key;
}

// Gate-weight fragments of batch b of this warp's (tile, part) units.
__device__ __forceinline__ void load_w_batch(const RouteArgs& a, int64_t kslice, int warp, int g, int t,
                                             int b, uint4 (&wv)[kRouteBatch][kRouteSpwMax]) {
#pragma unroll
    for (int uu = 0; uu < kRouteBatch; ++uu) {
        const int u = warp + kRouteWarps * (b * kRouteBatch + uu);
        const int j = u / a.wpt, p = u - j * a.wpt;
        const uint16_t* wp = a.w + (int64_t)(j * 8 + g) * a.K + kslice + (int64_t)p * a.spw * 32 + 8 * t;
#pragma unroll
        for (int s = 0; s < kRouteSpwMax; ++s)
            wv[uu][s] = (u < a.units && s < a.spw) ? ld_stream_v4(wp + s * 32) : make_uint4(0u, 0u, 0u, 0u);
    }
}

// Weights of the final selection (lane r < k holds slot r): identical
// arithmetic to the standalone gate kernel.
__device__ __forceinline__ float gate_weight(const RouteArgs& a, const float* row, float my_val) {
    const int lane = threadIdx.x & 31;
    const bool live = lane < a.topk;
    float num, den;
    if (a.scoring == 1) {
        num = live ? sigmoid_score(my_val) : 0.0f;
        den = a.renormalize ? warp_sum_fixed(num) : 1.0f;
        return a.renormalize ? __fdiv_rn(num, den) : num;
    }
    const float lmax = __shfl_sync(kFull, my_val, 0);
    num = live ? expf(__fadd_rn(my_val, -lmax)) : 0.0f;
    if (a.renormalize) {
        den = warp_sum_fixed(num);
    } else {
        float part = 0.0f;
        for (int id = lane; id < a.N; id += 32) part = __fadd_rn(part, expf(__fadd_rn(row[id], -lmax)));
        den = warp_sum_fixed(part);
    }
    return __fdiv_rn(num, den);
}

template <int MT, bool HALF>
__global__ void __launch_bounds__(kRouteThreads, 1) route_cluster_kernel(RouteArgs a) {
    extern __shared__ __align__(16) unsigned char sm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int c = (int)cluster_rank();
    MR_TRACE_STAMP(a.trace, 0);
    cluster_arrive_relaxed();  // completed by cluster_wait() before the first DSMEM store
    pdl_trigger();

    const int N = a.N, M = a.M, spw = a.spw, wpt = a.wpt, U = a.units, tok = a.tok;
    (void)spw;
    const int64_t kslice = (int64_t)c * a.kc;

    // ---- gate-weight loads of the first batch (the weight is never written
    //      by the preceding kernel, so they may precede the wait)
    uint4 wv[kRouteBatch][kRouteSpwMax];
    load_w_batch(a, kslice, warp, g, t, 0, wv);
    pdl_wait();

    // ---- x slice -> shared memory
    unsigned char* xs = sm + a.off_x;
    const int vpr = a.kc / 8;
    for (int v = tid; v < M * vpr; v += kRouteThreads) {
        const int r = v / vpr, cv = v - r * vpr;
        const uint4 d = ld_ro_v4(a.x + (int64_t)r * a.ldx + kslice + cv * 8);
        *reinterpret_cast<uint4*>(xs + r * a.xpitch + cv * 16) = d;
    }
    __syncthreads();
    MR_TRACE_STAMP(a.trace, 1);

    // ---- MXFP8 of the x slice (one lane quad per 32-block)
    if (a.q != nullptr) {
        const int nvec = M * vpr;
        const int64_t K32 = a.K / 32;
        for (int base = warp * 32; base < nvec; base += kRouteThreads) {
            const int v = base + lane;
            const int r = v / vpr, cv = v - r * vpr;
            const uint4 d = v < nvec ? lds128(xs + r * a.xpitch + cv * 16) : make_uint4(0u, 0u, 0u, 0u);
            unsigned sb;
            const uint2 q8 = mx_quant_quad(d, &sb);
            if (v < nvec) {
                const int64_t k = kslice + cv * 8;
                *reinterpret_cast<uint2*>(a.q + (int64_t)r * a.K + k) = q8;
                if ((cv & 3) == 0) a.scale[(int64_t)r * K32 + k / 32] = (uint8_t)sb;
            }
        }
    }

    // ---- MMA units; partial tiles straight to their owners' receive buffers
    cluster_wait();  // every CTA of the cluster is running: DSMEM is live
    const uint32_t recv_local = smem_u32(sm + a.off_recv);
    const int nb = (U - warp + kRouteWarps * kRouteBatch - 1) / (kRouteWarps * kRouteBatch);
    for (int b = 0; b < nb; ++b) {
        if (b > 0) load_w_batch(a, kslice, warp, g, t, b, wv);
#pragma unroll
        for (int uu = 0; uu < kRouteBatch; ++uu) {
            const int u = warp + kRouteWarps * (b * kRouteBatch + uu);
            if (u >= U) break;
            const int j = u / wpt, p = u - j * wpt;
            float acc[MT][4];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.0f;
#pragma unroll
            for (int s = 0; s < kRouteSpwMax; ++s) {
                if (s < spw) {
                    const int kk = (p * spw + s) * 32 + 8 * t;
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        const int r0 = mt * 16 + g, r1 = r0 + 8;
                        const uint4 xa = r0 < M ? lds128(xs + r0 * a.xpitch + kk * 2) : make_uint4(0u, 0u, 0u, 0u);
                        const uint4 xb = (!HALF && r1 < M) ? lds128(xs + r1 * a.xpitch + kk * 2)
                                                           : make_uint4(0u, 0u, 0u, 0u);
                        mma_bf16_m16n8k16(acc[mt], xa.x, xb.x, xa.y, xb.y, wv[uu][s].x, wv[uu][s].y);
                        mma_bf16_m16n8k16(acc[mt], xa.z, xb.z, xa.w, xb.w, wv[uu][s].z, wv[uu][s].w);
                    }
                }
            }
            const int col = j * 8 + 2 * t;
            const int slot = c * wpt + p;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                for (int h = 0; h < (HALF ? 1 : 2); ++h) {
                    const int r = mt * 16 + g + 8 * h;
                    if (r < M) {
                        const int own = r / tok, rl = r - own * tok;
                        const uint32_t la = recv_local + (uint32_t)(((slot * tok + rl) * N + col) * 4);
                        st_cluster_f2(map_rank(la, (unsigned)own), acc[mt][2 * h], acc[mt][2 * h + 1]);
                    }
                }
            }
        }
    }
    cluster_sync_acq_rel();  // barrier 1: every partial has reached its owner
    MR_TRACE_STAMP(a.trace, 2);

    // ---- owner: fixed-order split-K sum -> logits
    const float* recv = reinterpret_cast<const float*>(sm + a.off_recv);
    float* rowbuf = reinterpret_cast<float*>(sm + a.off_row);
    const int nslots = a.cs * wpt;
    const int my_rows = max(0, min(tok, M - c * tok));
    for (int idx = tid; idx < my_rows * N; idx += kRouteThreads) {
        const int rl = idx / N, n = idx - rl * N;
        const float* p = recv + (int64_t)rl * N + n;
        float s = 0.0f;
        for (int sl = 0; sl < nslots; ++sl) s = __fadd_rn(s, p[(int64_t)sl * tok * N]);
        rowbuf[idx] = s;
        a.logits[(int64_t)(c * tok + rl) * N + n] = s;
    }
    if (a.mode == 0) return;  // GEMV only: nothing else reads this CTA's memory
    __syncthreads();
    MR_TRACE_STAMP(a.trace, 3);

    // ---- gate: warp (row rl, segment sg) selects within experts [128 sg, 128 sg + 128)
    const int G = a.gwarps;
    unsigned* ckey = reinterpret_cast<unsigned*>(sm + a.off_cand);
    int* cid = reinterpret_cast<int*>(ckey + tok * G * 32);
    float* cval = reinterpret_cast<float*>(cid + tok * G * 32);
    const uint32_t ids_all_local = smem_u32(sm + a.off_ids);
    {
        const int rl = warp / G, sg = warp - rl * G;
        if (rl < my_rows) {
            const float* row = rowbuf + rl * N;
            unsigned key[4];
            int id[4];
            float val[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int e = sg * 128 + lane + 32 * jj;
                id[jj] = e;
                val[jj] = e < N ? row[e] : 0.0f;
                float sel = val[jj];
                if (a.scoring == 1 && e < N)
                    sel = __fadd_rn(sigmoid_score(val[jj]), a.bias ? __ldg(a.bias + e) : 0.0f);
                key[jj] = e < N ? ordered_key(sel) : 0u;
            }
            const int seg_len = max(0, min(128, N - sg * 128));
            const int kk = min(a.topk, seg_len);
            int my_id;
            float my_val;
            unsigned my_key;
            warp_select<4>(key, id, val, kk, &my_id, &my_val, &my_key);
            if (G == 1) {
                const float wgt = gate_weight(a, row, my_val);
                if (lane < a.topk) {
                    const int m = c * tok + rl;
                    a.ids[(int64_t)m * a.topk + lane] = my_id;
                    a.weights[(int64_t)m * a.topk + lane] = wgt;
                    st_cluster_s32(map_rank(ids_all_local + (uint32_t)((m * a.topk + lane) * 4), 0u), my_id);
                }
            } else {
                const int o = (rl * G + sg) * 32 + lane;
                ckey[o] = lane < kk ? my_key : 0u;
                cid[o] = lane < kk ? my_id : 0x7FFFFFFF - lane;
                cval[o] = my_val;
            }
        }
    }
    if (G > 1) {
        __syncthreads();
        const int rl = warp;  // one merging warp per row
        if (rl < my_rows) {
            unsigned key[8];
            int id[8];
            float val[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int sg = jj, o = (rl * G + sg) * 32 + lane;
                const bool ok = sg < G;
                key[jj] = ok ? ckey[o] : 0u;
                id[jj] = ok ? cid[o] : 0x7FFFFFFF - 32 * jj - lane;
                val[jj] = ok ? cval[o] : 0.0f;
            }
            int my_id;
            float my_val;
            unsigned my_key;
            warp_select<8>(key, id, val, a.topk, &my_id, &my_val, &my_key);
            const float wgt = gate_weight(a, rowbuf + rl * N, my_val);
            if (lane < a.topk) {
                const int m = c * tok + rl;
                a.ids[(int64_t)m * a.topk + lane] = my_id;
                a.weights[(int64_t)m * a.topk + lane] = wgt;
                st_cluster_s32(map_rank(ids_all_local + (uint32_t)((m * a.topk + lane) * 4), 0u), my_id);
            }
        }
    }
    cluster_sync_acq_rel();  // barrier 2: CTA 0 holds every token's ids
    MR_TRACE_STAMP(a.trace, 4);
    if (c != 0) return;

    // ---- sort (CTA 0): token bitmask per expert
    const int* ids_all = reinterpret_cast<const int*>(sm + a.off_ids);
    unsigned long long* mask = reinterpret_cast<unsigned long long*>(sm + a.off_mask);
    int* start = reinterpret_cast<int*>(sm + a.off_start);
    int* warp_tot = start + N;
    const int MK = M * a.topk, B = a.block;
    for (int e = tid; e < N; e += kRouteThreads) mask[e] = 0ull;
    __syncthreads();
    for (int f = tid; f < MK; f += kRouteThreads) atomicOr(&mask[ids_all[f]], 1ull << (f / a.topk));
    __syncthreads();
    for (int e = tid; e < N; e += kRouteThreads) start[e] = (__popcll(mask[e]) + B - 1) / B * B;
    __syncthreads();
    const int total = block_exclusive_scan(start, N, warp_tot);
    for (int f = tid; f < MK; f += kRouteThreads) {
        const int e = ids_all[f], m = f / a.topk;
        const int rank = __popcll(mask[e] & ((1ull << m) - 1ull));
        a.sorted[start[e] + rank] = f;
    }
    for (int e = tid; e < N; e += kRouteThreads) {
        const int st = start[e], cnt = __popcll(mask[e]), pad = (cnt + B - 1) / B * B;
        for (int i = cnt; i < pad; ++i) a.sorted[st + i] = MK;
        for (int b = st / B; b < (st + pad) / B; ++b) a.expert_ids[b] = e;
    }
    for (int64_t i = total + tid; i < a.capacity; i += kRouteThreads) a.sorted[i] = MK;
    for (int64_t b = total / B + tid; b < a.capacity / B; b += kRouteThreads) a.expert_ids[b] = -1;
    if (tid == 0) *a.ntpp = total;
    MR_TRACE_STAMP(a.trace, 5);
}

// ------------------------------------------------------------------ host

static int g_cluster16[64];     // per device: 0 unknown, 1 usable, -1 not
static int g_attr_done[64][4];  // per device and instantiation

template <int MT, bool HALF>
static cudaError_t prepare(int dev, int idx, int cs) {
    if (g_attr_done[dev][idx]) return cudaSuccess;
    auto k = route_cluster_kernel<MT, HALF>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kRouteSmemMax);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess) g_attr_done[dev][idx] = 1;
    (void)cs;
    return e;
}

int route_cluster_size() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 8;
    if (g_cluster16[dev] == 0) {
        cudaError_t e = prepare<1, false>(dev, 1, 16);
        int n = 0;
        if (e == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(16);
            cfg.blockDim = dim3(kRouteThreads);
            cfg.dynamicSmemBytes = kRouteSmemMax;
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = 16;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            e = cudaOccupancyMaxActiveClusters(&n, route_cluster_kernel<1, false>, &cfg);
        }
        g_cluster16[dev] = (e == cudaSuccess && n >= 1) ? 1 : -1;
        cudaGetLastError();  // a refused query leaves no sticky error
    }
    return g_cluster16[dev] > 0 ? 16 : 8;
}

cudaError_t launch_route_cluster(const RoutePlan& p, const RouteArgs& a, cudaStream_t st) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const int idx = p.half ? 0 : (p.mt == 1 ? 1 : p.mt == 2 ? 2 : 3);
    void (*kernel)(RouteArgs) = nullptr;
    switch (idx) {
        case 0: e = prepare<1, true>(dev, 0, p.cs); kernel = route_cluster_kernel<1, true>; break;
        case 1: e = prepare<1, false>(dev, 1, p.cs); kernel = route_cluster_kernel<1, false>; break;
        case 2: e = prepare<2, false>(dev, 2, p.cs); kernel = route_cluster_kernel<2, false>; break;
        default: e = prepare<4, false>(dev, 3, p.cs); kernel = route_cluster_kernel<4, false>; break;
    }
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.cs);
    cfg.blockDim = dim3(kRouteThreads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = p.cs;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = (launch_flags() & 1) ? 1 : 0;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kernel, a);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mr
