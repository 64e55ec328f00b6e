// The whole decode route in one launch for 1 <= M <= 16 tokens (a6).
//
// sglang #46691 (Summary) describes a one-launch decode router for 1-16
// tokens that is bitwise equal to the router GEMV, the gate and the sort run
// separately, and a sort + stage-1 quant in one launch for decode batches.
// Here the four steps share one grid:
//   * every CTA computes a split-K GEMV tile (same tiling and code as the
//     standalone GEMV, hence the same bits); the CTAs of n-block 0 also
//     quantise the x fragments they loaded (each element exactly once);
//   * the last CTA of each n-block (ticket 1) sums the partials in split
//     order and writes the logits;
//   * the last n-block to complete (ticket 2) runs the gate for all tokens,
//     one warp per token, and then sorts their assignments in the same CTA.
// Hand-offs are atomic last-arriver tickets, never spin-waits, so the launch
// completes whatever the residency of its CTAs.  Counters end at zero.
#include "gemv.cuh"
#include "gemv_configs.h"
#include "internal.h"
#include "sort.cuh"
#include "topk.cuh"

namespace mr {

struct FusedArgs {
    GemvArgs g;
    TopkArgs t;
    SortArgs s;
    uint8_t* q;
    uint8_t* scale;
    unsigned* done_counter;
};

template <class C, int NPL>
__global__ void __launch_bounds__(C::NTHR) fused_route_kernel(FusedArgs f) {
    extern __shared__ __align__(16) int sm[];
    __shared__ unsigned s_ticket;
    MR_TRACE_STAMP(f.g.trace, 0);
    pdl_trigger();
    const int nblk = blockIdx.x % f.g.nblocks, split = blockIdx.x / f.g.nblocks;
    QuantOut qo{f.q, f.scale};
    const bool quant_here = f.q != nullptr && nblk == 0;
    if (!gemv_cta<C>(f.g, nblk, split, 0, reinterpret_cast<float*>(sm), &s_ticket,
                     quant_here ? &qo : nullptr))
        return;
    const unsigned t = cta_ticket(f.done_counter, &s_ticket);
    MR_TRACE_STAMP(f.g.trace, 4);
    if (t != (unsigned)(f.g.nblocks - 1)) return;

    // gate of every token, then the sort, in this CTA
    const int N = f.g.N, n_assign = f.s.n_assign;
    RankSmem rs{sm, sm + C::NWARPS * N, sm + C::NWARPS * N + N};
    int* start = rs.lrank + n_assign;
    int* warp_tot = start + N;
    int* ids_s = warp_tot + 32;
    cta_topk_rows<NPL>(f.t, 0, f.g.M, ids_s);
    __syncthreads();
    MR_TRACE_STAMP(f.g.trace, 5);
    cta_sort(f.s, ids_s, rs, start, warp_tot);
    if (threadIdx.x == 0) *f.done_counter = 0u;
    MR_TRACE_STAMP(f.g.trace, 6);
}

template <class C>
static cudaError_t launch_fused_cfg(const FusedArgs& f, int npl, int nthr, cudaStream_t st) {
    const int n_assign = f.s.n_assign, N = f.g.N;
    const int sort_ints = C::NWARPS * N + 2 * N + n_assign + 32 + n_assign;
    const int smem = 4 * (sort_ints > C::RED_FLOATS ? sort_ints : C::RED_FLOATS);
    dim3 grid(f.g.nblocks * f.g.split_k);
    switch (npl) {
        case 4: return launch_kernel(fused_route_kernel<C, 4>, grid, dim3(nthr), smem, st, f);
        case 8: return launch_kernel(fused_route_kernel<C, 8>, grid, dim3(nthr), smem, st, f);
        case 16: return launch_kernel(fused_route_kernel<C, 16>, grid, dim3(nthr), smem, st, f);
        default: return launch_kernel(fused_route_kernel<C, 32>, grid, dim3(nthr), smem, st, f);
    }
}

// Only the M <= 8 and M <= 16 rows of the tiling table carry a fused kernel.
template <int I, class C>
static cudaError_t launch_fused_row(const FusedArgs& f, int npl, int nthr, cudaStream_t st) {
    if constexpr (I == MR_GEMV_CFG_M8 || I == MR_GEMV_CFG_M16)
        return launch_fused_cfg<C>(f, npl, nthr, st);
    else
        return cudaErrorInvalidValue;
}

cudaError_t launch_fused(const GemvPlan& p, const void* x, int64_t ldx, const void* w, int M,
                         int N, int K, int topk, int scoring, const float* bias,
                         int renormalize, int block, float* logits, int32_t* ids,
                         float* weights, int32_t* sorted, int32_t* expert_ids, int32_t* ntpp,
                         int64_t capacity, uint8_t* q, uint8_t* scale, void* scratch,
                         cudaStream_t st) {
    FusedArgs f;
    f.g.x = static_cast<const uint16_t*>(x);
    f.g.ldx = ldx;
    f.g.w = static_cast<const uint16_t*>(w);
    f.g.logits = logits;
    f.g.partials = reinterpret_cast<float*>(static_cast<char*>(scratch) + kWorkOffset);
    f.g.counters = static_cast<unsigned*>(scratch);
    f.g.M = M;
    f.g.N = N;
    f.g.K = K;
    f.g.split_k = p.split_k;
    f.g.nblocks = p.nblocks;
    f.g.trace = static_cast<unsigned long long*>(trace_buffer());
    f.t = TopkArgs{logits, bias, ids, weights, M, N, topk, scoring, renormalize};
    f.s = SortArgs{ids, M * topk, N, block, sorted, expert_ids, ntpp, capacity};
    f.q = q;
    f.scale = scale;
    f.done_counter = static_cast<unsigned*>(scratch) + kFusedCounterSlot;
    const int npl = topk_npl(N);
    switch (p.cfg) {
#define MR_FUSED_ROW(I, MT, HALF, NW, KW, KS) \
    case I:                                   \
        return launch_fused_row<I, GemvCfg<MT, HALF, NW, KW, KS>>(f, npl, p.nthr, st);
        MR_GEMV_CONFIGS(MR_FUSED_ROW)
#undef MR_FUSED_ROW
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace mr
