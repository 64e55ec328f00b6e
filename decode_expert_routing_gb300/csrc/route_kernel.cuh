// The decode route in ONE launch for M <= 64: router GEMV, split-K
// reduction, top-k gate, sort and MXFP8 (or MXFP4) quant.
//
// The pages' one-launch decode router (sglang #46691 Summary: a router for
// 1-16 tokens bitwise equal to router GEMV, gate and sort; sort + stage-1
// quant in one launch) chains its stages through global memory.  On GB300 a
// global last-arriver ticket costs ~0.7 us and a DSMEM message ~0.2 us, so
// this kernel keeps the hand-offs of up to 16 tokens inside one cluster of CS
// CTAs (16 when the device allows it, else 8):
//
//   1. CTA c owns the K slice [c*K/CS, (c+1)*K/CS) for ALL experts.  Warps
//      take (8-expert tile, k-part) units and run m16n8k16 bf16 MMAs with
//      fp32 accumulation; gate-weight fragments come straight from global
//      memory with 16-byte loads issued before the kernel waits on its
//      predecessor (programmatic dependent launch), x fragments from the
//      CTA's x slice in shared memory.
//   2. Split-K reduction: the WPT k-parts of a tile are added inside the
//      CTA (through shared memory, in part order), and the CTA's partial tile
//      goes by st.async to the CTA that owns the tile's token rows (token m
//      belongs to CTA m / TOK), counted on that CTA's mbarrier; the owner
//      waits for the bytes it expects and sums the CS partials of each logit
//      in CTA order.
//   3. Gate, the owner's whole CTA per row: a threshold below the k-th
//      largest key from group maxima, then a parallel ranking of the few
//      candidates; the chosen ids go at once to the sorting CTA (st.async).
//   4. The sorting CTA (one that owns no row when there is one, else CTA 0)
//      sorts the assignments: since the k ids of a token are distinct, the
//      stable rank of (m, j) inside expert e is popc(mask_e & ((1 << m) - 1))
//      where mask_e is the bitmask of the tokens that chose e.
//   More than 16 tokens: one cluster per 16 tokens, each running steps 1-3 on
//   its rows; the sorting CTAs publish their ids and take a last-arriver
//   ticket (the pages' hand-off), and the last one sorts every assignment.
//
// Variants of the same kernel:
//   - GEMV alone (mode 0): what the standalone router GEMV runs for
//     M <= 64, so the logits of the two are bitwise equal (above 64 rows the
//     tensor-core GEMV of kernel_tc_gemv.cu takes over).
//   - Expert groups (GROUPS, N >= 512): the experts split into groups of
//     >= 128, one cluster per group, so that more SMs share the gate weight;
//     for the whole route each cluster's collector publishes its group's
//     top-k candidates and the collector with the last ticket merges them.
//   - Route on the norm's scale (rstd != nullptr): x holds the residual rows
//     and each CTA forms bf16((x * rstd) * s) as it stages its slice.
//   - MXFP4 instead of MXFP8 stage-1 codes (quant_fp4).
//
// Every wait for bytes from other CTAs is bounded in time and sets a device
// flag when it runs out.  One cluster leaves nothing in scratch; several
// clusters leave their ticket counter at zero again.
#pragma once
#include <type_traits>
#include "cluster.cuh"
#include "common.cuh"
#include "internal.h"
#include "route_plan.h"

namespace mr {

// Set when a bounded wait of the route kernel ran out (read by the host).
// One per translation unit that instantiates the kernel (no separate device
// linking): each reports its own through route_timeout_flag below.
static __device__ int g_route_timeout;

// Thread 0 waits for phase 0 of the local mbarrier, at most limit_ns; the
// whole CTA learns the outcome (the barrier orders the data for every thread).
__device__ __forceinline__ bool cta_wait_bytes(uint32_t bar, unsigned long long limit_ns, int* s_ok) {
    if (threadIdx.x == 0) {
        bool ok = mbar_try_wait0(bar);
        if (!ok) {
            const unsigned long long t0 = global_ns();
            while (!(ok = mbar_try_wait0(bar)) && global_ns() - t0 < limit_ns) {
            }
            if (!ok) atomicExch(&g_route_timeout, 1);
        }
        *s_ok = ok ? 1 : 0;
    }
    __syncthreads();
    return *s_ok != 0;
}
// Barrier of the nthreads threads (whole warps) that use barrier id (1..15).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ uint4 lds128(const void* p) {
    return *reinterpret_cast<const uint4*>(p);
}
// x / d for 0 <= x < 2^21 with mag = ceil(2^32 / d) (host-computed)
__device__ __forceinline__ int fdiv(int x, unsigned long long mag) {
    return (int)(((unsigned long long)(unsigned)x * mag) >> 32);
}

// Gate-weight fragments of batch b of this warp's units.  A warp keeps one
// k-part p = warp % wpt for all its units, so the x fragments it loads serve
// every unit of a batch; unit i of the warp is tile (warp / wpt) + i * (16 / wpt).
__device__ __forceinline__ void load_w_batch(const RouteArgs& a, const uint16_t* wg, int64_t kslice, int warp,
                                             int g, int t, int b, uint4 (&wv)[kRouteBatch][kRouteSpwMax]) {
    const int p = warp & (a.wpt - 1), tiles_per_pass = kRouteWarps >> a.wpt_shift;
#pragma unroll
    for (int uu = 0; uu < kRouteBatch; ++uu) {
        const int j = (warp >> a.wpt_shift) + tiles_per_pass * (b * kRouteBatch + uu);
        const bool ok = j < (a.N >> 3);
        const uint16_t* wp = wg + (int64_t)(j * 8 + g) * a.K + kslice + (int64_t)p * a.spw * 32 + 8 * t;
#pragma unroll
        for (int s = 0; s < kRouteSpwMax; ++s)
            wv[uu][s] = (ok && s < a.spw) ? ld_stream_v4(wp + s * 32) : make_uint4(0u, 0u, 0u, 0u);
    }
}

// The MMAs of one batch over a k-part of SPW 32-wide steps (SPW = 0: spw
// at run time, at most kRouteSpwMax).  The kernel is instantiated per step
// count for the common hidden sizes (spw 6: K = 3072 / 6144 / 12288 on 16
// CTAs; 7: K = 3584 / 7168), each in its own translation unit: straight-line
// code the compiler schedules freely measured 0.12-0.24 us faster per launch
// than the run-time bound (a run-time switch between the variants inside
// one kernel kept only half of that: the kernel's code grew by 4-6 KB).
// xrow: this lane's x fragment of step 0 (step s at + 64 s bytes).
// At most 8 token rows: experts on the 16-row side, tokens on the 8 columns.
template <int SPW>
__device__ __forceinline__ void mma_steps_half(float (&acc)[4], float (&acc2)[4],
                                               const uint4 (&wv)[kRouteBatch][kRouteSpwMax],
                                               const unsigned char* xrow, bool live, int spw) {
#pragma unroll
    for (int s = 0; s < (SPW ? SPW : kRouteSpwMax); ++s) {
        if (SPW || s < spw) {
            const uint4 xa = live ? lds128(xrow + s * 64) : make_uint4(0u, 0u, 0u, 0u);
            mma_bf16_m16n8k16(acc, wv[0][s].x, wv[1][s].x, wv[0][s].y, wv[1][s].y, xa.x, xa.y);
            mma_bf16_m16n8k16(acc2, wv[0][s].z, wv[1][s].z, wv[0][s].w, wv[1][s].w, xa.z, xa.w);
        }
    }
}
// Up to 16 token rows: tokens on the 16-row side (rows g and g + 8), the
// batch's 8-expert tiles on the 8 columns; consecutive MMAs go to different
// accumulators.
template <int SPW>
__device__ __forceinline__ void mma_steps_full(float (&acc)[kRouteBatch][4],
                                               const uint4 (&wv)[kRouteBatch][kRouteSpwMax],
                                               const unsigned char* xrow0, const unsigned char* xrow1, bool live0,
                                               bool live1, int spw) {
#pragma unroll
    for (int s = 0; s < (SPW ? SPW : kRouteSpwMax); ++s) {
        if (SPW || s < spw) {
            const uint4 xa = live0 ? lds128(xrow0 + s * 64) : make_uint4(0u, 0u, 0u, 0u);
            const uint4 xb = live1 ? lds128(xrow1 + s * 64) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int uu = 0; uu < kRouteBatch; ++uu)
                mma_bf16_m16n8k16(acc[uu], xa.x, xb.x, xa.y, xb.y, wv[uu][s].x, wv[uu][s].y);
#pragma unroll
            for (int uu = 0; uu < kRouteBatch; ++uu)
                mma_bf16_m16n8k16(acc[uu], xa.z, xb.z, xa.w, xb.w, wv[uu][s].z, wv[uu][s].w);
        }
    }
}

// Selection order as one 64-bit integer: larger key first, then lower id.
__device__ __forceinline__ unsigned long long composite(unsigned key, int id) {
    return ((unsigned long long)key << 32) | (unsigned)(0x7FFFFFFF - id);
}

// Instantiations of the route kernel by what a launch computes.
constexpr int kKindGemv = 0, kKindSoftmax = 1, kKindSigmoid = 2;

// Weight of slot r = lane (lane < k holds (val) of slot r: its logit, or
// for the sigmoid gate (SIG) its exact score): the same arithmetic as the
// standalone gate kernel.  row: the token's n_row logits (only the
// full-softmax denominator reads it), in shared memory, or in global memory
// written by other CTAs (read through L2).
template <bool SIG>
__device__ __forceinline__ float gate_weight(const RouteArgs& a, const float* row, int n_row, bool global_row,
                                             float my_val) {
    const int lane = threadIdx.x & 31;
    const bool live = lane < a.topk;
    float num, den;
    if constexpr (SIG) {
        num = live ? my_val : 0.0f;
        den = a.renormalize ? warp_sum_fixed(num) : 1.0f;
        return a.renormalize ? __fdiv_rn(num, den) : num;
    }
    const float lmax = __shfl_sync(kFull, my_val, 0);
    num = live ? expf(__fadd_rn(my_val, -lmax)) : 0.0f;
    if (a.renormalize) {
        den = warp_sum_fixed(num);
    } else {
        float part = 0.0f;
        for (int id = lane; id < n_row; id += 32)
            part = __fadd_rn(part, expf(__fadd_rn(global_row ? __ldcg(row + id) : row[id], -lmax)));
        den = warp_sum_fixed(part);
    }
    return __fdiv_rn(num, den);
}

// MXFP8 (or MXFP4) of this CTA's x slice (rows row0 .. row0 + Mq, columns
// kslice .. kslice + kc), one lane quad per 32-element block; every thread of
// the CTA takes part.  The MXFP4 loop is one out-of-line copy: inlined at
// every call site beside the MXFP8 loop it made the kernel's code larger,
// and launches with a cold instruction cache measured 0.4-0.9 us slower.
// (The launch values are read once, on entry: through the reference the
// compiler would read them again after every store.)
static __device__ __noinline__ void quant_slice_fp4(const RouteArgs& a, const unsigned char* xs, int Mq,
                                                    int row0, int64_t kslice) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int vpr = a.kc / 8, nvec = Mq * vpr, xpitch = a.xpitch;
    const int64_t K = a.K, K32 = K / 32;
    const unsigned long long mag_vpr = a.mag_vpr;
    uint8_t* const q = a.q;
    uint8_t* const scale = a.scale;
    for (int base = warp * 32; base < nvec; base += kRouteThreads) {
        const int v = base + lane;
        const int r = fdiv(v, mag_vpr), cv = v - r * vpr;
        const uint4 d = v < nvec ? lds128(xs + r * xpitch + cv * 16) : make_uint4(0u, 0u, 0u, 0u);
        unsigned sb;
        const int64_t kk = kslice + cv * 8;
        const uint32_t q4 = mx4_quant_quad(d, &sb);
        if (v < nvec) *reinterpret_cast<uint32_t*>(q + (int64_t)(row0 + r) * (K / 2) + kk / 2) = q4;
        if (v < nvec && (cv & 3) == 0) scale[(int64_t)(row0 + r) * K32 + kk / 32] = (uint8_t)sb;
    }
}

__device__ __forceinline__ void quant_slice(const RouteArgs& a, const unsigned char* xs, int Mq, int row0,
                                            int64_t kslice) {
    if (a.q == nullptr) return;
    if (a.quant_fp4) {
        quant_slice_fp4(a, xs, Mq, row0, kslice);
        return;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int vpr = a.kc / 8, nvec = Mq * vpr;
    const int64_t K = a.K, K32 = K / 32;
    for (int base = warp * 32; base < nvec; base += kRouteThreads) {
        const int v = base + lane;
        const int r = fdiv(v, a.mag_vpr), cv = v - r * vpr;
        const uint4 d = v < nvec ? lds128(xs + r * a.xpitch + cv * 16) : make_uint4(0u, 0u, 0u, 0u);
        unsigned sb;
        const int64_t kk = kslice + cv * 8;
        const uint2 q8 = mx_quant_quad(d, &sb);
        if (v < nvec) *reinterpret_cast<uint2*>(a.q + (int64_t)(row0 + r) * K + kk) = q8;
        if (v < nvec && (cv & 3) == 0) a.scale[(int64_t)(row0 + r) * K32 + kk / 32] = (uint8_t)sb;
    }
}

// Sentinel MK in every slot of sorted_token_ids and -1 in every block of
// expert_ids (the sort then writes the real entries); all threads take part.
__device__ __forceinline__ void fill_sort_padding(const RouteArgs& a, int MK) {
    const int tid = threadIdx.x, cap = (int)a.capacity;  // < 2^31, checked on the host
    if ((reinterpret_cast<uintptr_t>(a.sorted) & 15u) == 0) {
        int4* st4 = reinterpret_cast<int4*>(a.sorted);
        const int n4 = cap >> 2;
        for (int i = tid; i < n4; i += kRouteThreads) st4[i] = make_int4(MK, MK, MK, MK);
        for (int i = (n4 << 2) + tid; i < cap; i += kRouteThreads) a.sorted[i] = MK;
    } else {
        for (int i = tid; i < cap; i += kRouteThreads) a.sorted[i] = MK;
    }
    for (int bb = tid, be = cap / a.block; bb < be; bb += kRouteThreads) a.expert_ids[bb] = -1;
}

// Gate weights of the CTA's owned rows: warp 15 - rl handles row rl.
template <bool SIG>
__device__ __forceinline__ void row_weights(const RouteArgs& a, const float* rowbuf, const float* oval, int my_rows,
                                            int grow) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, k = a.topk;
    if (warp >= kRouteWarps - my_rows) {
        const int rl = kRouteWarps - 1 - warp;
        const bool live = lane < k;
        const float wgt = gate_weight<SIG>(a, rowbuf + rl * a.N, a.N, false, live ? oval[rl * k + lane] : 0.0f);
        if (live) a.weights[(int64_t)(grow + rl) * k + lane] = wgt;
    }
}

// Shared expert's gate/up projection and SwiGLU, run by the clusters after
// the route's in the same launch (sglang #46691 Summary: the router fused
// with the shared expert's fp8 SwiGLU; sgl-amd-mono #56: the shared expert
// on its MXFP8 values with bf16 activations).  Cluster sc takes pairs
// [sc P, (sc + 1) P): local rows [0, P) are gate rows pair0 + i, rows
// [P, 2P) the up rows I + pair0 + i.  CTA c takes the K slice c for all of
// them, as the route does for the experts: warps run m16n8k16 bf16 MMAs on
// (8-row tile, k-part) units, the E4M3 weights converted to bf16 exactly
// and each 32-wide k step (one MX block) scaled by its E8M0 factor after
// its two MMAs (acc += block sum * 2^X, one fused multiply-add).  Partial
// sums go by st.async to the CTA that owns the token row, which adds the
// split-K partials in a fixed order and writes bf16(silu(gate) * up).
// Out of line (inlined, it made every cold launch of the route ~2 us
// slower); it reads each launch value it needs once, on entry.
template <int SPW>  // 32-wide k steps per k-part, as the route's (0: a.sh_spw at run time)
static __device__ __noinline__ void shared_gate_up_cta(const RouteArgs& a, int sc) {
    extern __shared__ __align__(16) unsigned char sm[];
    __shared__ __align__(8) unsigned long long s_shbar, s_shwbar;  // partials in; weight rows in
    __shared__ int s_shok;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t = lane & 3;
    const int c = (int)cluster_rank();
    // every launch value this function uses, read once here (through the
    // reference the compiler would read some again after every store)
    const int Mq = a.M, K = a.K, kc = a.kc, P = a.sh_pairs, R = 2 * P, I = a.sh_I;
    const int tok = a.tok, wpt = a.sh_wpt, spw = SPW ? SPW : a.sh_spw, nslots = a.sh_nslots;
    const int xpitch = a.xpitch, units = a.sh_units, tok_shift = a.tok_shift, spitch = a.sh_spitch;
    const int flags = a.flags;
    const unsigned long long wait_ns = a.wait_ns;
    const int64_t ldx = a.ldx;
    const uint16_t* const xg = a.x;
    const uint16_t* const norm_w = a.norm_w;
    const float* const rstd = a.rstd;
    const bool gemma = a.norm_gemma != 0;
    const uint8_t* const wg8 = a.sh_w;
    const uint8_t* const sg8 = a.sh_scale;
    uint16_t* const out = a.sh_out;
    unsigned char* const ws = sm + a.sh_off_w;
    unsigned char* const ss = sm + a.sh_off_s;
    unsigned char* const xs = sm + a.sh_off_x;
    const uint32_t recv_local = smem_u32(sm + a.sh_off_recv);
    const int my_rows = max(0, min(tok, Mq - c * tok));
    const int pair0 = sc * P;
    const uint32_t bar = smem_u32(&s_shbar), wbar = smem_u32(&s_shwbar);
    const int wpitch = kc + 16, spr = kc / 32;
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(wbar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        const unsigned stall = (flags & 2) ? 16u : 0u;  // test hook: bytes that never come
        if (my_rows > 0) mbar_expect_tx(bar, (unsigned)(my_rows * nslots * R * 4) + stall);
        mbar_expect_tx(wbar, (unsigned)(R * kc));
    }
    cluster_arrive_relaxed();
    pdl_trigger();
    const int64_t kslice = (int64_t)c * kc;
    const int K32 = K / 32;
    // The CTA's weight slice (R rows x kc E4M3 bytes, rows padded by 16 B
    // against bank conflicts) goes to shared memory by bulk copies, a row
    // each (kc bytes, a multiple of 32; K a multiple of 512 and the base
    // 16-byte aligned, so every row starts on a 16-byte boundary), counted on
    // wbar; its scale bytes by plain loads; all issued before the dependency
    // wait (they are parameters).  Then units u = warp, warp + 16, ... (tile
    // j = u / wpt, k-part p = u % wpt) read them from there in a rolled loop
    // (a CTA runs it once, from a cold instruction cache).
    __syncthreads();  // wbar initialised before any copy counts on it
    for (int lr = tid; lr < R; lr += kRouteThreads) {
        const int64_t gr = lr < P ? pair0 + lr : I + pair0 + (lr - P);
        bulk_load(smem_u32(ws + lr * wpitch), wg8 + gr * K + kslice, (unsigned)kc, wbar);
    }
    if (tid < R) {  // a thread per row: its kc / 32 scale bytes, 8 loads in flight at a time
        const int64_t gr = tid < P ? pair0 + tid : I + pair0 + (tid - P);
        const uint8_t* src = sg8 + gr * K32 + kslice / 32;
        for (int b0 = 0; b0 < spr; b0 += 8) {
            uint8_t v[8];
#pragma unroll
            for (int b = 0; b < 8; ++b) v[b] = b0 + b < spr ? __ldg(src + b0 + b) : 0;
#pragma unroll
            for (int b = 0; b < 8; ++b)
                if (b0 + b < spr) ss[tid * spitch + b0 + b] = v[b];
        }
    }
    pdl_wait();
    // the x slice -> shared memory (on the norm's scale when rstd is given),
    // as f16 when every value of the CTA's slice converts exactly: then the
    // E4M3 weights go to the MMAs by one conversion per pair (f16 holds every
    // E4M3 value) instead of the longer exact E4M3 -> bf16 one, and the
    // products and their fp32 sums are those of the bf16 MMAs.  Otherwise
    // (a value at or above 2^16 or below 2^-17) the slice is staged again as
    // bf16 and the bf16 MMAs run.
    const int vpr = kc / 8;
    bool exact = true;
    for (int v = tid; v < Mq * vpr; v += kRouteThreads) {
        const int r = v / vpr, cv = v - r * vpr;
        uint4 d = ld_ro_v4(xg + (int64_t)r * ldx + kslice + cv * 8);
        if (rstd != nullptr) d = norm_chunk(d, ld_ro_v4(norm_w + kslice + cv * 8), __ldg(rstd + r), gemma);
        d = make_uint4(bf16x2_to_f16x2(d.x, &exact), bf16x2_to_f16x2(d.y, &exact), bf16x2_to_f16x2(d.z, &exact),
                       bf16x2_to_f16x2(d.w, &exact));
        *reinterpret_cast<uint4*>(xs + r * xpitch + cv * 16) = d;
    }
    // thread 0 waits for the weight rows (bounded: after a wait that ran out
    // it sets the flag and waits once more, so that no copy is left in
    // flight; the CTA then goes on, its partials not valid, so that its
    // owners' waits and its own still end)
    if (tid == 0) {
        bool ok = mbar_try_wait0(wbar);
        if (!ok) {
            unsigned long long t0 = global_ns();
            while (!(ok = mbar_try_wait0(wbar)) && global_ns() - t0 < wait_ns) {
            }
            if (!ok) {
                atomicExch(&g_route_timeout, 1);
                t0 = global_ns();
                while (!mbar_try_wait0(wbar) && global_ns() - t0 < wait_ns) {
                }
            }
        }
    }
    const bool use_f16 = __syncthreads_and(exact) != 0;
    if (!use_f16) {
        for (int v = tid; v < Mq * vpr; v += kRouteThreads) {
            const int r = v / vpr, cv = v - r * vpr;
            uint4 d = ld_ro_v4(xg + (int64_t)r * ldx + kslice + cv * 8);
            if (rstd != nullptr) d = norm_chunk(d, ld_ro_v4(norm_w + kslice + cv * 8), __ldg(rstd + r), gemma);
            *reinterpret_cast<uint4*>(xs + r * xpitch + cv * 16) = d;
        }
        __syncthreads();
    }
    cluster_wait();  // every CTA of the cluster is running: DSMEM is live
    uint32_t owner_bar[2] = {0u, 0u};
#pragma unroll
    for (int h = 0; h < 2; ++h)
        if (g + 8 * h < Mq) owner_bar[h] = map_rank(bar, (unsigned)((g + 8 * h) >> tok_shift));
    // one (tile, k-part) unit: each 32-wide k step (one MX block) is two MMAs
    // into a fresh block sum, added to the accumulator times its E8M0 scale
    auto unit_steps = [&](auto f16, int j, int p, float (&acc)[4]) {
        constexpr bool F16 = decltype(f16)::value;
        const unsigned char* wrow = ws + (j * 8 + g) * wpitch + p * spw * 32 + 8 * t;
        const unsigned char* srow0 = ss + (j * 8 + 2 * t) * spitch + p * spw;
#pragma unroll
        for (int s = 0; s < (SPW ? SPW : kRouteSpwMax); ++s) {
            if (SPW || s < spw) {
                const int kk = (p * spw + s) * 32 + 8 * t;
                const uint4 xa = g < Mq ? lds128(xs + g * xpitch + kk * 2) : make_uint4(0u, 0u, 0u, 0u);
                const uint4 xb = g + 8 < Mq ? lds128(xs + (g + 8) * xpitch + kk * 2) : make_uint4(0u, 0u, 0u, 0u);
                const uint2 w8 = *reinterpret_cast<const uint2*>(wrow + s * 32);
                float blk[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                if constexpr (F16) {
                    const uint32_t b0 = e4m3x2_to_f16x2(w8.x), b1 = e4m3x2_to_f16x2(w8.x >> 16);
                    const uint32_t b2 = e4m3x2_to_f16x2(w8.y), b3 = e4m3x2_to_f16x2(w8.y >> 16);
                    mma_f16_m16n8k16(blk, xa.x, xb.x, xa.y, xb.y, b0, b1);
                    mma_f16_m16n8k16(blk, xa.z, xb.z, xa.w, xb.w, b2, b3);
                } else {
                    const uint32_t b0 = e4m3x2_to_bf16x2(w8.x), b1 = e4m3x2_to_bf16x2(w8.x >> 16);
                    const uint32_t b2 = e4m3x2_to_bf16x2(w8.y), b3 = e4m3x2_to_bf16x2(w8.y >> 16);
                    mma_bf16_m16n8k16(blk, xa.x, xb.x, xa.y, xb.y, b0, b1);
                    mma_bf16_m16n8k16(blk, xa.z, xb.z, xa.w, xb.w, b2, b3);
                }
                const float s0 = e8m0_value(srow0[s]), s1 = e8m0_value(srow0[spitch + s]);
                acc[0] = __fmaf_rn(blk[0], s0, acc[0]);
                acc[1] = __fmaf_rn(blk[1], s1, acc[1]);
                acc[2] = __fmaf_rn(blk[2], s0, acc[2]);
                acc[3] = __fmaf_rn(blk[3], s1, acc[3]);
            }
        }
    };
#pragma unroll 1
    for (int u = warp; u < units; u += kRouteWarps) {
        const int j = u / wpt, p = u - j * wpt;
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (use_f16)
            unit_steps(std::true_type{}, j, p, acc);
        else
            unit_steps(std::false_type{}, j, p, acc);
        const int col = j * 8 + 2 * t, slot = c * wpt + p;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = g + 8 * h;
            if (r < Mq) {
                const int own = r >> tok_shift, rl = r & (tok - 1);
                const uint32_t la = recv_local + (uint32_t)(((slot * tok + rl) * R + col) * 4);
                st_async_f2(map_rank(la, (unsigned)own), acc[2 * h], acc[2 * h + 1], owner_bar[h]);
            }
        }
    }
    if (my_rows == 0) return;
    if (!cta_wait_bytes(bar, wait_ns, &s_shok)) return;
    // owner: pair i of each owned row; partials added in slot order
    const float* recv = reinterpret_cast<const float*>(sm + (recv_local - smem_u32(sm)));
    const int plane = tok * R;
    for (int idx = tid; idx < my_rows * P; idx += kRouteThreads) {
        const int rl = idx / P, i = idx - rl * P;
        const float* pg = recv + rl * R + i;
        float gs = 0.0f, us = 0.0f;
        for (int sl = 0; sl < nslots; sl += 8) {
            float vg[8], vu[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                vg[q] = pg[(sl + q) * plane];
                vu[q] = pg[(sl + q) * plane + P];
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                gs = __fadd_rn(gs, vg[q]);
                us = __fadd_rn(us, vu[q]);
            }
        }
        const float act = __fmul_rn(__fdiv_rn(gs, __fadd_rn(1.0f, expf(-gs))), us);
        uint16_t b;
        asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(b) : "f"(act));
        out[(int64_t)(c * tok + rl) * I + pair0 + i] = b;
    }
}

// HALF: at most 8 token rows (half of the m16 tile live).
// GROUPS: the experts are split into a.ng groups, one cluster per group.
// KIND: kKindGemv (mode 0, the GEMV alone), kKindSoftmax or kKindSigmoid
// (mode 1 with that gate).  Each its own instantiation, carrying only its
// code: the sigmoid gate's exact scoring is a third of the route's code,
// and carried unexecuted by the softmax kernel it made every cold launch
// ~3 us slower (a warm one ~0.15 us); the GEMV alone needs half the code of
// the route.
// SH: the launch carries the shared expert's clusters (after the route's, or
// alone).  Their CTA code is ~22 KB, a quarter of the softmax route's code
// and half of the GEMV alone's, so only these instantiations carry it.
template <bool HALF, bool GROUPS, int KIND, bool SH, int SPW>
__global__ void __launch_bounds__(kRouteThreads, 1) route_cluster_kernel(RouteArgs a) {
    constexpr bool SIG = KIND == kKindSigmoid, GEMV = KIND == kKindGemv;
    extern __shared__ __align__(16) unsigned char sm[];
    __shared__ __align__(8) unsigned long long s_bar[3];  // [0] partial logits in, [1] ids in, [2] MMAs done
    __shared__ int s_ok[3];
    __shared__ unsigned s_ticket;
    __shared__ __align__(16) unsigned s_wmin[kRouteWarps];  // gate: per warp, smallest group maximum
    __shared__ int s_ccount;                                  // gate: candidates so far
    __shared__ __align__(16) int s_wtot[2 * kRouteWarps];     // sort: blocks per warp (experts t, t + 512)
    if constexpr (SH) {
        if ((int)(blockIdx.x >> a.cs_shift) >= a.clusters) {  // the shared expert's clusters
            shared_gate_up_cta<SPW>(a, (int)(blockIdx.x >> a.cs_shift) - a.clusters);
            return;
        }
    }
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int c = (int)cluster_rank();
    MR_TRACE_STAMP(a.trace, 0);
#ifdef MR_TRACE
    if (tid == 0 && a.trace) a.trace[blockIdx.x * 512 + 24] = clock64();
#endif
    // this cluster's token rows: [row0, row0 + Mq); this CTA owns rows
    // [c * tok, c * tok + my_rows) of them
    // expert groups: cluster cl takes token group cl / ng and experts
    // [e_off, e_off + N) of ldn (its group, nc = cl % ng)
    const int cl = (int)(blockIdx.x >> a.cs_shift);
    const int mc = GROUPS ? cl / a.ng : cl, nc = GROUPS ? cl - mc * a.ng : 0;
    const int row0 = mc * a.rpc;
    const int Mq = min(a.rpc, a.M - row0);
    const int N = a.N, wpt = a.wpt, tok = a.tok, K = a.K, k = a.topk;
    const int nslots = a.nslots;
    const int my_rows = max(0, min(tok, Mq - c * tok));
    // the CTA that sorts the cluster's assignments: one that owns no row when
    // there is one (it is idle while the others run the gate), else CTA 0
    const int sorter = Mq <= (a.cs - 1) * tok ? a.cs - 1 : 0;
    // (with expert groups it collects the cluster's group candidates, and
    // the last cluster's collector merges and sorts)
    const bool sorts = !GEMV && c == sorter;
    const bool quants = nc == 0;  // one expert group per token group quantises x
    const int e_off = GROUPS ? nc * N : 0;
    const uint32_t bar0 = smem_u32(&s_bar[0]), bar1 = smem_u32(&s_bar[1]), bar2 = smem_u32(&s_bar[2]);
    if (tid == 0) {
        s_ccount = 0;
        mbar_init(bar0, 1);
        mbar_init(bar1, 1);
        mbar_init(bar2, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        const unsigned stall = (a.flags & 2) ? 16u : 0u;  // test hook: bytes that never come
        if (my_rows > 0) mbar_expect_tx(bar0, (unsigned)(my_rows * nslots * N * 4) + stall);
        if (sorts) mbar_expect_tx(bar1, (unsigned)(Mq * k * (GROUPS ? 12 : 4)));
    }
    cluster_arrive_relaxed();  // completed by cluster_wait() before the first DSMEM access
    pdl_trigger();
    {   // Every launch gets a fresh copy of its parameters in constant memory:
        // touch each 32-byte line of it now, so that no later phase stalls on
        // a first-use miss.
        const unsigned long long acc =
            (unsigned long long)a.x ^ (unsigned long long)a.logits ^ (unsigned long long)a.expert_ids ^
            (unsigned long long)a.scale ^ (unsigned long long)a.renormalize ^ (unsigned long long)a.units ^
            (unsigned long long)a.off_ids ^ a.mag_n ^ (unsigned long long)a.trace ^ (unsigned long long)a.counter ^
            (unsigned long long)a.norm_gemma;
        asm volatile("" ::"l"(acc));
    }
    const int64_t kslice = (int64_t)c * a.kc;
    const uint16_t* xq = a.x + (int64_t)row0 * a.ldx;
    const uint16_t* wg = a.w + (int64_t)e_off * K;  // this cluster's expert rows
    unsigned long long* mask = reinterpret_cast<unsigned long long*>(sm + a.off_mask);

    // ---- loads of the gate weight (first batch) and of the selection bias:
    //      parameters, never written by the preceding kernel, so they may
    //      precede the wait
    uint4 wv[kRouteBatch][kRouteSpwMax];
    const int vpr = a.kc / 8;  // 16-byte chunks per row of the CTA's K slice
    load_w_batch(a, wg, kslice, warp, g, t, 0, wv);
    float bpre0 = 0.0f, bpre1 = 0.0f;  // selection bias of this thread's experts t and t + 512
    if (a.bias != nullptr) {
        if (tid < N) bpre0 = __ldg(a.bias + e_off + tid);
        if (tid + kRouteThreads < N) bpre1 = __ldg(a.bias + e_off + tid + kRouteThreads);
    }
    if (sorts)
        for (int e = tid; e < N; e += kRouteThreads) mask[e] = 0ull;  // token bitmasks (2 x 32 bits per expert)
    pdl_wait();
    MR_TRACE_STAMP(a.trace, 8);

    // ---- this CTA's x slice -> shared memory (on the norm's scale: the
    //      residual rows times rstd and the norm weight, rounded to bf16 as
    //      the norm would store them)
    unsigned char* xs = sm + a.off_x;
    const bool norm = a.rstd != nullptr;
    if (norm) {
        for (int v = tid; v < Mq * vpr; v += kRouteThreads) {
            const int r = fdiv(v, a.mag_vpr), cv = v - r * vpr;
            uint4 d = ld_ro_v4(xq + (int64_t)r * a.ldx + kslice + cv * 8);
            d = norm_chunk(d, ld_ro_v4(a.norm_w + kslice + cv * 8), __ldg(a.rstd + row0 + r), a.norm_gemma != 0);
            *reinterpret_cast<uint4*>(xs + r * a.xpitch + cv * 16) = d;
        }
    } else {  // straight to shared memory: every chunk in flight at once, no register round trip
        for (int v = tid; v < Mq * vpr; v += kRouteThreads) {
            const int r = fdiv(v, a.mag_vpr), cv = v - r * vpr;
            cp_async16(smem_u32(xs + r * a.xpitch + cv * 16), xq + (int64_t)r * a.ldx + kslice + cv * 8);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    MR_TRACE_WARP(a.trace, 0);
    __syncthreads();
    MR_TRACE_STAMP(a.trace, 1);

    // ---- MMA: batches of units sharing one k-part; partial tiles go
    //      straight to the receive buffers of the rows' owners
    cluster_wait();  // every CTA of the cluster is running: DSMEM is live
    const uint32_t recv_local = smem_u32(sm + a.off_recv);
    uint32_t owner_bar[2] = {0u, 0u};  // mbarrier of the owner of rows g and g + 8
#pragma unroll
    for (int h = 0; h < 2; ++h)
        if (g + 8 * h < Mq) owner_bar[h] = map_rank(bar0, (unsigned)((g + 8 * h) >> a.tok_shift));
    const int p = warp & (wpt - 1), tiles_per_pass = kRouteWarps >> a.wpt_shift, NT = N >> 3;
    const int j0 = warp >> a.wpt_shift;
    const int my_tiles = j0 < NT ? (NT - j0 + tiles_per_pass - 1) >> (4 - a.wpt_shift) : 0;
    const int nb = (my_tiles + kRouteBatch - 1) / kRouteBatch;
    // The warps of one tile group (its wpt k-parts) add their partial tiles
    // before sending: parts p >= 1 leave theirs in shared memory (one buffer
    // per batch parity), and after the group's barrier part 0 adds them in
    // part order and sends one partial per CTA and logit (slot c).
    float* const kred = reinterpret_cast<float*>(sm + a.off_kred);
    const int kbar = 1 + j0, kthreads = 32 * wpt;
    const int slot = c;
    const int r0 = g, r1 = g + 8;  // one m16 tile: at most 16 token rows per cluster here
    // this lane's x fragments of step 0 of its k-part: row g (the HALF
    // path's one token column, else the MMA's row g) and row g + 8
    const unsigned char* xrow0 = xs + r0 * a.xpitch + ((p * a.spw) * 32 + 8 * t) * 2;
    const unsigned char* xrow1 = xrow0 + 8 * a.xpitch;
    uint32_t tok_bar[2] = {0u, 0u};  // at most 8 rows: mbarrier of the owner of tokens 2t and 2t + 1
#pragma unroll
    for (int h = 0; h < 2; ++h)
        if (2 * t + h < Mq) tok_bar[h] = map_rank(bar0, (unsigned)((2 * t + h) >> a.tok_shift));
    for (int b = 0; b < nb; ++b) {
        if (b > 0) load_w_batch(a, wg, kslice, warp, g, t, b, wv);
        if constexpr (HALF) {
            // At most 8 token rows: the experts take the MMA's 16-row side
            // (the batch's two 8-expert tiles, rows 0-7 and 8-15) and the
            // tokens its 8 columns, so one pair of MMAs per 32-wide k step
            // covers both tiles (half the MMAs of tokens on the 16-row side,
            // where 8 of the 16 rows are empty).
            static_assert(kRouteBatch == 2, "two 8-expert tiles make the 16 rows");
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f}, acc2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            mma_steps_half<SPW>(acc, acc2, wv, xrow0, g < Mq, SPW ? SPW : a.spw);
            MR_TRACE_WARP(a.trace, 4);
            // acc[2 uu + h]: the expert of row g of unit uu's tile, token 2t + h
            float v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = __fadd_rn(acc[i], acc2[i]);
            if (wpt > 1) {
                float* kb = kred + (b & 1) * (kRouteWarps * 4 * 32);
                if (p != 0) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) kb[(warp * 4 + i) * 32 + lane] = v[i];
                }
                named_bar_sync(kbar, kthreads);
                if (p != 0) continue;
                for (int q = 1; q < wpt; ++q) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) v[i] = __fadd_rn(v[i], kb[((warp + q) * 4 + i) * 32 + lane]);
                }
            }
#pragma unroll
            for (int uu = 0; uu < 2; ++uu) {
                const int j = j0 + tiles_per_pass * (b * 2 + uu);
                if (j >= NT) break;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = 2 * t + h;
                    if (r < Mq) {
                        const int own = r >> a.tok_shift, rl = r & (tok - 1);
                        const uint32_t la = recv_local + (uint32_t)(((slot * tok + rl) * N + j * 8 + g) * 4);
                        st_async_s32(map_rank(la, (unsigned)own), __float_as_int(v[2 * uu + h]), tok_bar[h]);
                    }
                }
            }
            continue;
        }
        float acc[kRouteBatch][4];
#pragma unroll
        for (int uu = 0; uu < kRouteBatch; ++uu) acc[uu][0] = acc[uu][1] = acc[uu][2] = acc[uu][3] = 0.0f;
        mma_steps_full<SPW>(acc, wv, xrow0, xrow1, r0 < Mq, !HALF && r1 < Mq, SPW ? SPW : a.spw);
        MR_TRACE_WARP(a.trace, 4);
        if (wpt > 1) {
            float* kb = kred + (b & 1) * (kRouteWarps * 8 * 32);
            if (p != 0) {
#pragma unroll
                for (int uu = 0; uu < kRouteBatch; ++uu)
#pragma unroll
                    for (int i = 0; i < 4; ++i) kb[(warp * 8 + uu * 4 + i) * 32 + lane] = acc[uu][i];
            }
            named_bar_sync(kbar, kthreads);
            if (p != 0) continue;
            for (int q = 1; q < wpt; ++q) {
#pragma unroll
                for (int uu = 0; uu < kRouteBatch; ++uu)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        acc[uu][i] = __fadd_rn(acc[uu][i], kb[((warp + q) * 8 + uu * 4 + i) * 32 + lane]);
            }
        }
#pragma unroll
        for (int uu = 0; uu < kRouteBatch; ++uu) {
            const int j = j0 + tiles_per_pass * (b * kRouteBatch + uu);
            if (j >= NT) break;
            const int col = j * 8 + 2 * t;
#pragma unroll
            for (int h = 0; h < (HALF ? 1 : 2); ++h) {
                const int r = g + 8 * h;
                if (r < Mq) {
                    const int own = r >> a.tok_shift, rl = r & (tok - 1);
                    const uint32_t la = recv_local + (uint32_t)(((slot * tok + rl) * N + col) * 4);
                    st_async_f2(map_rank(la, (unsigned)own), acc[uu][2 * h], acc[uu][2 * h + 1], owner_bar[h]);
                }
            }
        }
    }
    MR_TRACE_WARP(a.trace, 1);
    MR_TRACE_WARP(a.trace, 2);
    MR_TRACE_STAMP(a.trace, 12);
    // The sorter quantises its slice now (and, with one cluster, fills the
    // sentinels and the -1 block ids; the real entries overwrite them after
    // barriers of this CTA).  A CTA that owns no rows and does not sort is
    // done once its slice is quantised: nothing is ever sent to it.  Owners
    // quantise later, off the path of the gate.
    if (sorts) {
        if (!GEMV && quants) quant_slice(a, xs, Mq, row0, kslice);
        if (a.clusters == 1) fill_sort_padding(a, a.M * k);
    } else if (my_rows == 0) {
        if (!GEMV && quants) quant_slice(a, xs, Mq, row0, kslice);
        return;
    }
    if (my_rows > 0 && !cta_wait_bytes(bar0, a.wait_ns, &s_ok[0])) return;
    MR_TRACE_CLK(a.trace, 0);
    MR_TRACE_STAMP(a.trace, 2);

    // ---- per owned row: split-K sum, logits, gate.
    //      Owner sum: thread t sums expert t (and t + 512) over the split-K
    //      slots in a fixed order (the GEMV-only mode runs the same code).
    //      Gate: selection order is the 64-bit composite (key, ~id): unique,
    //      larger first.  Lane groups of GL = 2^gs_shift <= 32 threads hold
    //      disjoint expert sets, G >= k of them hold experts; T, the smallest
    //      group maximum key, has at least G >= k keys at or above it, so
    //      every top-k expert has key >= T.  The experts with key >= T
    //      (candidates) are ranked among themselves: a candidate's rank is
    //      the number of candidates that beat it.  The winners' ids go out at
    //      once (to CTA 0 for the sort, and to HBM).
    const float* recv = reinterpret_cast<const float*>(sm + a.off_recv);
    float* rowbuf = reinterpret_cast<float*>(sm + a.off_row);
    unsigned long long* ccand = reinterpret_cast<unsigned long long*>(sm + a.off_cand);
    float* oval = reinterpret_cast<float*>(ccand + N);  // per owned row: the k winners' values
    float* cscore = oval + tok * k;                     // sigmoid gate: exact score of candidate i
    const int grow = row0 + c * tok;  // global index of this CTA's first row
    const int plane = tok * N;        // floats between two slots of the receive buffer
    const int n0 = tid, n1 = tid + kRouteThreads;
    const bool h0 = n0 < N, h1 = n1 < N;
    const int gl = 1 << a.gs_shift;
    const unsigned gmask = gl == 32 ? kFull : ((1u << gl) - 1u) << (lane & ~(gl - 1));
    const bool group_has = (tid & ~(gl - 1)) < N;  // the lane group's first expert exists
    if constexpr (GEMV) {  // GEMV alone: every (owned row, expert) in parallel
        for (int idx = tid; idx < my_rows * N; idx += kRouteThreads) {
            const int rl = fdiv(idx, a.mag_n), n = idx - rl * N;
            const float* pp = recv + rl * N + n;
            float sum = 0.0f;
            for (int sl = 0; sl < nslots; sl += 8) {  // the same order as below
                float v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = pp[(sl + u) * plane];
#pragma unroll
                for (int u = 0; u < 8; ++u) sum = __fadd_rn(sum, v[u]);
            }
            a.logits[(int64_t)(grow + rl) * a.ldn + e_off + n] = sum;
        }
        MR_TRACE_STAMP(a.trace, 3);
        return;  // nothing else reads this CTA's shared memory
    }
    for (int rl = 0; rl < my_rows; ++rl) {
        float sum0 = 0.0f, sum1 = 0.0f;
        if (h0) {
            const float* pp = recv + rl * N + n0;
            if (nslots == 16) {  // every load in flight, then the adds in order
                float v[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) v[u] = pp[u * plane];
#pragma unroll
                for (int u = 0; u < 16; ++u) sum0 = __fadd_rn(sum0, v[u]);
            } else {
                for (int sl = 0; sl < nslots; sl += 8) {  // nslots % 8 == 0; loads first, then the adds in order
                    float v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) v[u] = pp[(sl + u) * plane];
#pragma unroll
                    for (int u = 0; u < 8; ++u) sum0 = __fadd_rn(sum0, v[u]);
                }
            }
        }
        if (h1) {
            const float* pp = recv + rl * N + n1;
            for (int sl = 0; sl < nslots; sl += 8) {
                float v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = pp[(sl + u) * plane];
#pragma unroll
                for (int u = 0; u < 8; ++u) sum1 = __fadd_rn(sum1, v[u]);
            }
        }
        const int64_t lrow = (int64_t)(grow + rl) * a.ldn + e_off;
        if (h0) {
            rowbuf[rl * N + n0] = sum0;
            a.logits[lrow + n0] = sum0;
        }
        if (h1) {
            rowbuf[rl * N + n1] = sum1;
            a.logits[lrow + n1] = sum1;
        }
        float sel0 = sum0, sel1 = sum1;
        if constexpr (SIG) {  // approximate keys: they only pick the candidates
            sel0 = __fadd_rn(sigmoid_approx(sum0), bpre0);
            sel1 = __fadd_rn(sigmoid_approx(sum1), bpre1);
        }
        const unsigned long long c0 = h0 ? composite(ordered_key(sel0), e_off + n0) : 0ull;
        const unsigned long long c1 = h1 ? composite(ordered_key(sel1), e_off + n1) : 0ull;
        const unsigned k0 = (unsigned)(c0 >> 32), k1 = (unsigned)(c1 >> 32);
        // the warp's smallest maximum over its groups that hold experts
        const unsigned gmax = __reduce_max_sync(gmask, max(k0, k1));
        const unsigned wx = __reduce_min_sync(kFull, group_has ? gmax : 0xFFFFFFFFu);
        if (lane == 0) s_wmin[warp] = wx;
        MR_TRACE_CLK(a.trace, 1);
        __syncthreads();  // s_wmin; rowbuf of this row
        MR_TRACE_CLK(a.trace, 3);
        unsigned T = __reduce_min_sync(kFull, lane < kRouteWarps ? s_wmin[lane] : 0xFFFFFFFFu);
        // sigmoid gate: every expert of the exact top-k has an approximate
        // key within the margin of the k-th largest (>= T), so the
        // candidates reach that far down
        if constexpr (SIG) T = sigmoid_candidate_floor(T);
        MR_TRACE_CLK(a.trace, 4);
        const bool p0 = h0 && k0 >= T, p1 = h1 && k1 >= T;
        const unsigned b0 = __ballot_sync(kFull, p0), b1 = __ballot_sync(kFull, p1);
        const int wc = __popc(b0) + __popc(b1);
        int base = 0;
        if (lane == 0 && wc != 0) base = atomicAdd(&s_ccount, wc);
        base = __shfl_sync(kFull, base, 0);
        const unsigned lt = (1u << lane) - 1u;
        if (p0) ccand[base + __popc(b0 & lt)] = c0;
        if (p1) ccand[base + __popc(b0) + __popc(b1 & lt)] = c1;
        __syncthreads();
        MR_TRACE_CLK(a.trace, 5);
        // PR adjacent lanes per candidate, each counting the beaters among
        // candidates part, part + PR, ...; a segmented reduction adds them
        const int C = s_ccount;
        if constexpr (SIG) {  // the candidates' exact scores and keys (correctly rounded sigmoid + bias)
            for (int i = tid; i < C; i += kRouteThreads) {
                const int id = 0x7FFFFFFF - (int)(unsigned)(ccand[i] & 0xFFFFFFFFull);
                const float b = a.bias != nullptr ? __ldg(a.bias + id) : 0.0f;
                const float sc = sigmoid_exact(rowbuf[rl * N + id - e_off], (a.flags & 8) != 0);
                cscore[i] = sc;
                ccand[i] = composite(ordered_key(__fadd_rn(sc, b)), id);
            }
            __syncthreads();
        }
        int prs = 5;
        while (prs > 0 && (C << prs) > kRouteThreads) --prs;
        const int PR = 1 << prs;
        const unsigned pmask = PR == 32 ? kFull : ((1u << PR) - 1u) << (lane & ~(PR - 1));
        const int ml = c * tok + rl, m = grow + rl;
        for (int base2 = warp * 32; base2 < (C << prs); base2 += kRouteThreads) {
            const int item = base2 + lane, ci = item >> prs, part = item & (PR - 1);
            if (ci < C) {  // whole segments of PR lanes
                const unsigned long long cn = ccand[ci];
                int r = 0;
                for (int j = part; j < C; j += PR) r += (int)(ccand[j] > cn);
                r = (int)__reduce_add_sync(pmask, (unsigned)r);
                if (GROUPS && part == 0 && r < k) {  // the group's r-th candidate -> the collector
                    const int id = 0x7FFFFFFF - (int)(unsigned)(cn & 0xFFFFFFFFull);
                    const uint32_t cb = smem_u32(sm + a.off_merge), sbar = map_rank(bar1, (unsigned)sorter);
                    st_async_f2(map_rank(cb + (uint32_t)((ml * k + r) * 8), (unsigned)sorter),
                                __uint_as_float((unsigned)cn), __uint_as_float((unsigned)(cn >> 32)), sbar);
                    const float v = SIG ? cscore[ci] : rowbuf[rl * N + id - e_off];
                    st_async_s32(map_rank(cb + (uint32_t)(Mq * k * 8 + (ml * k + r) * 4), (unsigned)sorter),
                                 __float_as_int(v), sbar);
                } else if (part == 0 && r < k) {
                    const int id = 0x7FFFFFFF - (int)(unsigned)(cn & 0xFFFFFFFFull);
                    st_async_s32(map_rank(smem_u32(sm + a.off_ids) + (uint32_t)((ml * k + r) * 4), (unsigned)sorter),
                                 id, map_rank(bar1, (unsigned)sorter));
                    a.ids[(int64_t)m * k + r] = id;
                    oval[rl * k + r] = SIG ? cscore[ci] : rowbuf[rl * N + id];
                }
            }
        }
        __syncthreads();  // oval complete; every thread has read s_ccount
        if (tid == 0) s_ccount = 0;  // before the next row's second barrier
    }
    MR_TRACE_WARP(a.trace, 3);
    MR_TRACE_STAMP(a.trace, 4);
    MR_TRACE_CLK(a.trace, 9);
    MR_TRACE_CLK(a.trace, 11);
    MR_TRACE_WARP(a.trace, 7);
    int* ids_all = reinterpret_cast<int*>(sm + a.off_ids);
    const int M = a.M, MK = M * k, B = a.block, NS = a.ldn;
    if constexpr (GROUPS) {
        // ---- expert groups: the owners have sent their rows' group
        //      candidates (k per row, in rank order) to the cluster's
        //      collector, which publishes them and takes a ticket; the last
        //      collector merges them into each token's top-k, writes the ids
        //      and weights, and sorts.  The merge ranks candidate (g, r) of
        //      token m by r plus, for every other group, the count of its
        //      candidates that beat it (a binary search: each list is
        //      descending; the composites are unique).
        if (!sorts) {
            if (!GEMV && quants) quant_slice(a, xs, Mq, row0, kslice);
            return;
        }
        if (!cta_wait_bytes(bar1, a.wait_ns, &s_ok[1])) return;
        MR_TRACE_STAMP(a.trace, 5);
        {
            const unsigned long long* ckey = reinterpret_cast<const unsigned long long*>(sm + a.off_merge);
            const float* cval = reinterpret_cast<const float*>(sm + a.off_merge + Mq * k * 8);
            for (int f = tid; f < Mq * k; f += kRouteThreads) {
                const int rr = fdiv(f, a.mag_k), j = f - rr * k;
                const int64_t slot = ((int64_t)(row0 + rr) * a.ng + nc) * k + j;
                a.cand_key[slot] = ckey[f];
                a.cand_val[slot] = cval[f];
            }
        }
        const unsigned ticket = cta_ticket(a.counter, &s_ticket);
        if (ticket != (unsigned)(a.clusters - 1)) return;
        // one warp per token: its ng lists of k candidates (each descending)
        // go to shared memory; lane g < ng holds the head of list g, and k
        // rounds each take the largest head (two redux.sync maximums: the
        // high words, then the low words among the lanes that tie on them;
        // the composites are unique, so one lane wins) and advance that list
        const int ngk = a.ng * k;
        unsigned long long* mkey = reinterpret_cast<unsigned long long*>(sm + a.off_merge);
        float* mval = reinterpret_cast<float*>(mkey + M * ngk);
        for (int e = tid; e < NS; e += kRouteThreads) mask[e] = 0ull;
        if (tid == 0) *a.counter = 0u;
        MR_TRACE_CLK(a.trace, 6);
        for (int m = warp; m < M; m += kRouteWarps) {
            unsigned long long* ck = mkey + m * ngk;
            float* cv = mval + m * ngk;
            {   // all loads in flight before the stores (ngk <= 8 * 32)
                unsigned long long kr[kRouteMaxGroups];
                float vr[kRouteMaxGroups];
#pragma unroll
                for (int q = 0; q < kRouteMaxGroups; ++q) {
                    const int i = lane + 32 * q;
                    if (i < ngk) {
                        kr[q] = __ldcg(a.cand_key + (int64_t)m * ngk + i);
                        vr[q] = __ldcg(a.cand_val + (int64_t)m * ngk + i);
                    }
                }
#pragma unroll
                for (int q = 0; q < kRouteMaxGroups; ++q) {
                    const int i = lane + 32 * q;
                    if (i < ngk) {
                        ck[i] = kr[q];
                        cv[i] = vr[q];
                    }
                }
            }
            __syncwarp();
            const bool owns = lane < a.ng;
            const unsigned long long* L = ck + lane * k;
            int ptr = 0;
            unsigned long long head = owns ? L[0] : 0ull;
            unsigned long long nxt = (owns && k > 1) ? L[1] : 0ull;
            float myval = 0.0f;  // lane r < k: the logit of slot r
            for (int r = 0; r < k; ++r) {
                const unsigned hi = (unsigned)(head >> 32);
                const unsigned mhi = __reduce_max_sync(kFull, hi);
                const unsigned mlo = __reduce_max_sync(kFull, hi == mhi ? (unsigned)head : 0u);
                const bool win = owns && hi == mhi && (unsigned)head == mlo;
                const unsigned wl = __ballot_sync(kFull, win);
                const float v = __shfl_sync(kFull, (owns && ptr < k) ? cv[lane * k + ptr] : 0.0f, __ffs(wl) - 1);
                if (lane == r) myval = v;
                if (win) {
                    const int id = 0x7FFFFFFF - (int)mlo;
                    ids_all[m * k + r] = id;
                    a.ids[(int64_t)m * k + r] = id;
                    ++ptr;
                    head = nxt;
                    nxt = ptr + 1 < k ? L[ptr + 1] : 0ull;
                }
            }
            MR_TRACE_CLK(a.trace, 7);
            const bool live = lane < k;
            const float wgt = gate_weight<SIG>(a, a.logits + (int64_t)m * NS, NS, true, live ? myval : 0.0f);
            if (live) a.weights[(int64_t)m * k + lane] = wgt;
        }
        __syncthreads();  // every token's ids; the masks zeroed
        MR_TRACE_CLK(a.trace, 8);
    } else {
    if (!sorts) {  // the weights and the quantisation finish this CTA
        row_weights<SIG>(a, rowbuf, oval, my_rows, grow);
        quant_slice(a, xs, Mq, row0, kslice);
        return;
    }
    row_weights<SIG>(a, rowbuf, oval, my_rows, grow);
    if (!cta_wait_bytes(bar1, a.wait_ns, &s_ok[1])) return;
    MR_TRACE_STAMP(a.trace, 5);
    MR_TRACE_WARP(a.trace, 9);

    // ---- sort.  One cluster: CTA 0 holds every id.  Several clusters: each
    //      CTA 0 publishes its rows' ids and takes a ticket; the last one
    //      gathers all ids and sorts (with several clusters its first phase
    //      also fills the sentinels and the -1 block ids).  HALF launches
    //      (at most 8 rows) without expert groups are one cluster: their
    //      instantiation carries none of this (about 10 KB of code).
    if (!HALF && a.clusters > 1) {
        for (int f = tid; f < Mq * k; f += kRouteThreads) a.ids_scratch[row0 * k + f] = ids_all[f];
        const unsigned ticket = cta_ticket(a.counter, &s_ticket);
        if (ticket != (unsigned)(a.clusters - 1)) return;
        // every row from scratch (this cluster's own ids sit at local offsets)
        {   // straight to shared memory, 16 bytes a copy (the tail by plain loads)
            const int n4 = MK >> 2;
            for (int i = tid; i < n4; i += kRouteThreads)
                cp_async16(smem_u32(ids_all + 4 * i), a.ids_scratch + 4 * i);
            asm volatile("cp.async.commit_group;" ::: "memory");
            for (int f = (n4 << 2) + tid; f < MK; f += kRouteThreads) ids_all[f] = __ldcg(a.ids_scratch + f);
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        if (tid == 0) *a.counter = 0u;
        __syncthreads();
    }
    }  // one expert group
    MR_TRACE_STAMP(a.trace, 6);
    MR_TRACE_CLK(a.trace, 13);
    // rank of (m, j) inside expert e = number of set bits below m in the token
    // mask of e (two 32-bit words: tokens 0-31, 32-63)
    int* start = reinterpret_cast<int*>(sm + a.off_start);
    unsigned* mlo = reinterpret_cast<unsigned*>(mask);
    unsigned* mhi = mlo + NS;
    for (int f = tid; f < MK; f += kRouteThreads) {
        const int m = fdiv(f, a.mag_k);
        atomicOr(m < 32 ? &mlo[ids_all[f]] : &mhi[ids_all[f]], 1u << (m & 31));
    }
    if ((GROUPS || !HALF) && a.clusters > 1) fill_sort_padding(a, MK);
    __syncthreads();
    MR_TRACE_CLK(a.trace, 14);
    MR_TRACE_WARP(a.trace, 10);
    MR_TRACE_CLK(a.trace, 15);
    // blocks per expert nb = ceil(count / B); thread t: experts t and t + 512.
    // Exclusive scan over the experts: inside a warp from the ballots of the
    // bits of nb (nb <= ceil(M / B) < 2^nbits), kept in start[]; across warps
    // from the 32 warp totals (experts 0..511 by warp, then 512..1023), which
    // every warp scans with shuffles after one barrier: lane i then holds the
    // blocks before the experts of total i, i = e / 32.  With no further
    // barrier, each expert's thread writes its real blocks' expert id (padding
    // blocks already hold -1) and each assignment's thread its slot of sorted
    // ids (the first block of its expert plus the expert's tokens before it).
    static_assert(2 * kRouteWarps == 32, "one warp total per lane");
    const int e0 = tid, e1 = tid + kRouteThreads;
    const int nb0 = e0 < NS ? fdiv(__popc(mlo[e0]) + __popc(mhi[e0]) + B - 1, a.mag_block) : 0;
    const int nb1 = e1 < NS ? fdiv(__popc(mlo[e1]) + __popc(mhi[e1]) + B - 1, a.mag_block) : 0;
    const int nbits = 32 - __clz(fdiv(M + B - 1, a.mag_block));
    const unsigned lt = (1u << lane) - 1u;
    int pre0 = 0, pre1 = 0, wt0 = 0, wt1 = 0;
    for (int bit = 0; bit < nbits; ++bit) {
        const unsigned q0 = __ballot_sync(kFull, (nb0 >> bit) & 1), q1 = __ballot_sync(kFull, (nb1 >> bit) & 1);
        pre0 += __popc(q0 & lt) << bit;
        pre1 += __popc(q1 & lt) << bit;
        wt0 += __popc(q0) << bit;
        wt1 += __popc(q1) << bit;
    }
    if (e0 < NS) start[e0] = pre0;
    if (e1 < NS) start[e1] = pre1;
    if (lane == 0) {
        s_wtot[warp] = wt0;
        s_wtot[kRouteWarps + warp] = wt1;
    }
    MR_TRACE_CLK(a.trace, 16);
    __syncthreads();  // start[] (in-warp prefixes) and the warp totals
    int wexc;         // lane i: blocks of the warp totals before total i
    {
        const int wv = s_wtot[lane];
        int inc = wv;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int o = __shfl_up_sync(kFull, inc, d);
            if (lane >= d) inc += o;
        }
        wexc = inc - wv;
        if (tid == 31) *a.ntpp = inc * B;
    }
    MR_TRACE_CLK(a.trace, 17);
    {
        const int sb0 = __shfl_sync(kFull, wexc, warp) + pre0;  // first block of e0
        if (e0 < NS)
            for (int i = 0; i < nb0; ++i) a.expert_ids[sb0 + i] = e0;
        const int sb1 = __shfl_sync(kFull, wexc, kRouteWarps + warp) + pre1;
        if (e1 < NS)
            for (int i = 0; i < nb1; ++i) a.expert_ids[sb1 + i] = e1;
    }
    MR_TRACE_CLK(a.trace, 19);
    MR_TRACE_WARP(a.trace, 12);
    MR_TRACE_CLK(a.trace, 22);
    for (int base = warp * 32; base < MK; base += kRouteThreads) {  // whole warps (shuffles)
        const int f = base + lane;
        const int e = f < MK ? ids_all[f] : 0, m = fdiv(f, a.mag_k);
        const int sb = __shfl_sync(kFull, wexc, e >> 5);
        if (f < MK) {
            const unsigned below = m < 32 ? __popc(mlo[e] & ((1u << m) - 1u))
                                          : __popc(mlo[e]) + __popc(mhi[e] & ((1u << (m - 32)) - 1u));
            a.sorted[(sb + start[e]) * B + (int)below] = f;
        }
    }
    MR_TRACE_CLK(a.trace, 23);
    MR_TRACE_WARP(a.trace, 13);
#ifdef MR_TRACE
    if (tid == 0 && a.trace) a.trace[blockIdx.x * 512 + 25] = clock64();
#endif
    MR_TRACE_STAMP(a.trace, 7);
}

// ------------------------------------------------------------------ host
// (static: one copy per translation unit that instantiates the kernel)

// this unit's bounded-wait flag (clear: reset it when set)
static int route_timeout_flag(int clear) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_route_timeout, sizeof(int)) != cudaSuccess) return -1;
    if (clear && v != 0) {
        const int z = 0;
        if (cudaMemcpyToSymbol(g_route_timeout, &z, sizeof(int)) != cudaSuccess) return -1;
    }
    return v;
}

static int g_attr_done[64][24];  // per device and instantiation

template <bool HALF, bool GROUPS, int KIND, bool SH, int SPW>
static cudaError_t prepare(int dev) {
    const int slot = (HALF ? 1 : 0) + (GROUPS ? 2 : 0) + 4 * KIND + (SH ? 12 : 0);
    if (g_attr_done[dev][slot]) return cudaSuccess;
    auto k = route_cluster_kernel<HALF, GROUPS, KIND, SH, SPW>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kRouteSmemMax);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess) g_attr_done[dev][slot] = 1;
    return e;
}

// The launch of plan p with the instantiation of step count SPW (the GEMV
// alone carrying the shared expert has no route clusters: SPW unused).
template <int SPW>
static cudaError_t launch_route_spw(const RoutePlan& p, const RouteArgs& a, cudaStream_t st) {

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    void (*kernel)(RouteArgs) = nullptr;
    const int kind = a.mode == 0 ? kKindGemv : (a.scoring == 1 ? kKindSigmoid : kKindSoftmax);
    const bool sh = p.sh_clusters > 0;
#define MR_ONE(H, G, K, S)                                \
    do {                                                  \
        e = prepare<H, G, K, S, SPW>(dev);                     \
        kernel = route_cluster_kernel<H, G, K, S, SPW>;        \
    } while (0)
#define MR_ROUTE(H, G)                                                        \
    do {                                                                      \
        if (kind == kKindSigmoid) {                                           \
            if (sh) MR_ONE(H, G, kKindSigmoid, true); else MR_ONE(H, G, kKindSigmoid, false); \
        } else {                                                              \
            if (sh) MR_ONE(H, G, kKindSoftmax, true); else MR_ONE(H, G, kKindSoftmax, false); \
        }                                                                     \
    } while (0)
    if (kind == kKindGemv) {
        // (the GEMV alone never carries the shared expert: with shared
        // clusters and no route clusters this is mr_shared_gate_up)
        if (sh) MR_ONE(false, false, kKindGemv, true);
        else if (p.ng > 1 && p.half) MR_ONE(true, true, kKindGemv, false);
        else if (p.ng > 1) MR_ONE(false, true, kKindGemv, false);
        else if (p.half) MR_ONE(true, false, kKindGemv, false);
        else MR_ONE(false, false, kKindGemv, false);
    } else if (p.ng > 1 && p.half) {
        MR_ROUTE(true, true);
    } else if (p.ng > 1) {
        MR_ROUTE(false, true);
    } else if (p.half) {
        MR_ROUTE(true, false);
    } else {
        MR_ROUTE(false, false);
    }
#undef MR_ROUTE
#undef MR_ONE
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.cs * (p.clusters + p.sh_clusters));
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
