// Split-K router GEMV tile and its in-kernel fixup.
//
// The method (sglang #36557, description): logits[M,N] = x[M,K] . W[N,K]^T
// with the K range split over CTAs; the last CTA to finish a (n-block,
// row-tile) pair reduces the SPLIT_K partials and resets its counter slot, so
// there is neither a zero-init launch nor a reduce launch.
//
// GB300 design.  A warp owns an 8-expert tile (the n8 side of an m16n8k16
// bf16 tensor-core MMA with fp32 accumulation) and KS consecutive 32-wide k
// steps.  Lane (g = lane/4, t = lane%4) reads the 16 contiguous bytes
// W[n0+g][k+8t .. k+8t+7] with one streaming 16-byte load; four lanes cover
// 64 contiguous bytes of a gate row, so every sector fetched is used.  The
// MMA's k order inside a 32-wide step is a permutation of the physical k
// (the dot product does not care), applied identically to x and W:
//   MMA 0 takes physical k {8t, 8t+1} (slot 2t..2t+1) and {8t+2, 8t+3}
//   (slot 2t+8..2t+9); MMA 1 takes {8t+4..8t+7} the same way.
// x rows g and g+8 of each 16-row tile load the same 16 bytes of their row,
// so the A fragment is two 16-byte loads per step with no shuffles.  All of
// a warp's loads are issued before its first MMA.  Partials of the KW warps
// along k are summed in warp order through shared memory; partials of the
// SPLIT_K CTAs are summed in split order by the last CTA.  Every expert n
// sees the same k partition and order, so bitwise-identical gate rows give
// bitwise-identical logits.
#pragma once

#include "common.cuh"

namespace mr {

struct GemvArgs {
    const uint16_t* x;     // bf16 [M, ldx]
    int64_t ldx;
    const uint16_t* w;     // bf16 [N, K]
    float* logits;         // fp32 [M, N]
    float* partials;       // fp32 [split_k, M, N]   (split_k > 1)
    unsigned* counters;    // [row_tiles * nblocks]
    int M, N, K;
    int split_k;           // CTAs along K
    int nblocks;           // N / BLOCK_N
    unsigned long long* trace;  // phase stamps (tracing builds only), or nullptr
};

// Where the fused kernel puts MXFP8 codes of the x fragments it loads.
struct QuantOut {
    uint8_t* q;            // [M, K]
    uint8_t* scale;        // [M, K/32]
};

template <int MT_, bool HALF_, int NW_, int KW_, int KS_>
struct GemvCfg {
    static constexpr int MT = MT_;        // 16-row tiles per CTA
    static constexpr bool HALF = HALF_;   // only rows 0..7 of the tile are live (M <= 8)
    static constexpr int NW = NW_;        // 8-expert tiles per CTA (warps along N)
    static constexpr int KW = KW_;        // warps along K
    static constexpr int KS = KS_;        // 32-wide k steps per warp
    static constexpr int NWARPS = NW * KW;
    static constexpr int NTHR = NWARPS * 32;
    static constexpr int BLOCK_N = 8 * NW;
    static constexpr int ROWS = 16 * MT;
    static constexpr int KCHUNK = 32 * KS * KW;
    // shared floats for the cross-warp reduction
    static constexpr int RED_FLOATS = (KW - 1) * NW * MT * 32 * 4;
};

// Computes the CTA tile (nblk, split, rt).  On return the lanes of the warps
// with wk == 0 hold the CTA's sums in acc: acc[mt][0..1] = rows r0, cols c, c+1;
// acc[mt][2..3] = rows r0 + 8, with r0 = rt*ROWS + mt*16 + lane/4 and
// c = nblk*BLOCK_N + wn*8 + 2*(lane%4).  If qo != nullptr the warps with
// wn == 0 also write the MXFP8 codes of the x they loaded.
template <class C>
__device__ __forceinline__ void gemv_tile(const GemvArgs& a, int nblk, int split, int rt,
                                          float (&acc)[C::MT][4], float* red,
                                          const QuantOut* qo) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int wn = warp % C::NW, wk = warp / C::NW;
    const int n = nblk * C::BLOCK_N + wn * 8 + g;
    const int64_t kbeg = (int64_t)split * C::KCHUNK + (int64_t)wk * (32 * C::KS) + 8 * t;

    uint4 wv[C::KS];
    const uint16_t* wrow = a.w + (int64_t)n * a.K + kbeg;
#pragma unroll
    for (int s = 0; s < C::KS; ++s) wv[s] = ld_stream_v4(wrow + s * 32);
    // The gate weight is never written by the preceding kernel; everything
    // else (x, scratch, outputs) is touched only after it has completed.
    pdl_wait();

    uint4 xa[C::MT][C::KS], xb[C::MT][C::KS];
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt) {
        const int r0 = rt * C::ROWS + mt * 16 + g, r1 = r0 + 8;
        const uint16_t* x0 = a.x + (int64_t)r0 * a.ldx + kbeg;
        const uint16_t* x1 = a.x + (int64_t)r1 * a.ldx + kbeg;
#pragma unroll
        for (int s = 0; s < C::KS; ++s) {
            xa[mt][s] = (r0 < a.M) ? ld_ro_v4(x0 + s * 32) : zero;
            xb[mt][s] = (!C::HALF && r1 < a.M) ? ld_ro_v4(x1 + s * 32) : zero;
        }
    }

    float c[C::MT][4];
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt) c[mt][0] = c[mt][1] = c[mt][2] = c[mt][3] = 0.0f;
#pragma unroll
    for (int s = 0; s < C::KS; ++s) {
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
            mma_bf16_m16n8k16(c[mt], xa[mt][s].x, xb[mt][s].x, xa[mt][s].y, xb[mt][s].y,
                              wv[s].x, wv[s].y);
            mma_bf16_m16n8k16(c[mt], xa[mt][s].z, xb[mt][s].z, xa[mt][s].w, xb[mt][s].w,
                              wv[s].z, wv[s].w);
        }
    }

    if (qo != nullptr && wn == 0) {
        const int K32 = a.K / 32;
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
            const int r0 = rt * C::ROWS + mt * 16 + g, r1 = r0 + 8;
#pragma unroll
            for (int s = 0; s < C::KS; ++s) {
                const int64_t k = kbeg + s * 32;  // = block start + 8t
                unsigned sb;
                uint2 q8 = mx_quant_quad(xa[mt][s], &sb);
                if (r0 < a.M) {
                    *reinterpret_cast<uint2*>(qo->q + (int64_t)r0 * a.K + k) = q8;
                    if (t == 0) qo->scale[(int64_t)r0 * K32 + k / 32] = (uint8_t)sb;
                }
                if (!C::HALF) {
                    q8 = mx_quant_quad(xb[mt][s], &sb);
                    if (r1 < a.M) {
                        *reinterpret_cast<uint2*>(qo->q + (int64_t)r1 * a.K + k) = q8;
                        if (t == 0) qo->scale[(int64_t)r1 * K32 + k / 32] = (uint8_t)sb;
                    }
                }
            }
        }
    }

    if constexpr (C::KW > 1) {
        if (wk > 0) {
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt) {
                float4* dst = reinterpret_cast<float4*>(red) +
                              (((wk - 1) * C::NW + wn) * C::MT + mt) * 32 + lane;
                *dst = make_float4(c[mt][0], c[mt][1], c[mt][2], c[mt][3]);
            }
        }
        __syncthreads();
        if (wk == 0) {
#pragma unroll
            for (int j = 1; j < C::KW; ++j) {
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) {
                    float4 v = reinterpret_cast<const float4*>(red)[(((j - 1) * C::NW + wn) * C::MT + mt) * 32 + lane];
                    c[mt][0] = __fadd_rn(c[mt][0], v.x);
                    c[mt][1] = __fadd_rn(c[mt][1], v.y);
                    c[mt][2] = __fadd_rn(c[mt][2], v.z);
                    c[mt][3] = __fadd_rn(c[mt][3], v.w);
                }
            }
        }
    }
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[mt][i] = c[mt][i];
}

// Stores the CTA sums held by the wk == 0 warps to dst [*, M, N] (dst =
// logits when the launch has a single split, else this split's partials).
template <class C>
__device__ __forceinline__ void gemv_store(const GemvArgs& a, float* dst, int nblk, int rt,
                                           const float (&acc)[C::MT][4]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int wn = warp % C::NW, wk = warp / C::NW;
    if (wk != 0) return;
    const int col = nblk * C::BLOCK_N + wn * 8 + 2 * t;
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt) {
        const int r0 = rt * C::ROWS + mt * 16 + g, r1 = r0 + 8;
        if (r0 < a.M)
            *reinterpret_cast<float2*>(dst + (int64_t)r0 * a.N + col) = make_float2(acc[mt][0], acc[mt][1]);
        if (!C::HALF && r1 < a.M)
            *reinterpret_cast<float2*>(dst + (int64_t)r1 * a.N + col) = make_float2(acc[mt][2], acc[mt][3]);
    }
}

// Full GEMV step for one CTA: tile, store, ticket, and (for the last CTA of
// the (n-block, row-tile) pair) the fixup.  Returns true in the CTA that
// completed the logits of its pair (always true when split_k == 1).
template <class C>
__device__ __forceinline__ bool gemv_cta(const GemvArgs& a, int nblk, int split, int rt,
                                         float* red, unsigned* s_ticket, const QuantOut* qo) {
    float acc[C::MT][4];
    gemv_tile<C>(a, nblk, split, rt, acc, red, qo);
    MR_TRACE_STAMP(a.trace, 1);
    if (a.split_k == 1) {
        gemv_store<C>(a, a.logits, nblk, rt, acc);
        return true;
    }
    gemv_store<C>(a, a.partials + (int64_t)split * a.M * a.N, nblk, rt, acc);
    unsigned* ctr = a.counters + rt * a.nblocks + nblk;
    const unsigned ticket = cta_ticket(ctr, s_ticket);
    MR_TRACE_STAMP(a.trace, 2);
    if (ticket != (unsigned)(a.split_k - 1)) return false;
    // fixup: sum the partials of every split in split order (loads of up to
    // 8 splits in flight at once, adds in order)
    const int rows = min(C::ROWS, a.M - rt * C::ROWS);
    const int64_t plane = (int64_t)a.M * a.N;
    for (int e = threadIdx.x; e < rows * C::BLOCK_N; e += C::NTHR) {
        const int r = rt * C::ROWS + e / C::BLOCK_N;
        const int col = nblk * C::BLOCK_N + e % C::BLOCK_N;
        const float* p = a.partials + (int64_t)r * a.N + col;
        float s = 0.0f;
        for (int sp0 = 0; sp0 < a.split_k; sp0 += 8) {
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = (sp0 + i < a.split_k) ? __ldcg(p + (sp0 + i) * plane) : 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (sp0 + i < a.split_k) s = __fadd_rn(s, v[i]);
        }
        a.logits[(int64_t)r * a.N + col] = s;
    }
    if (threadIdx.x == 0) *ctr = 0u;
    MR_TRACE_STAMP(a.trace, 3);
    return true;
}

}  // namespace mr
