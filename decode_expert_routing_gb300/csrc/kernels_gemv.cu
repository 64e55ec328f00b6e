// Router GEMV launch (a1 + a2): split-K tiles with the in-kernel fixup.
#include "gemv.cuh"
#include "gemv_configs.h"
#include "internal.h"

namespace mr {

template <class C>
__global__ void __launch_bounds__(C::NTHR) router_gemv_kernel(GemvArgs a) {
    __shared__ __align__(16) float red[C::RED_FLOATS > 0 ? C::RED_FLOATS : 4];
    __shared__ unsigned s_ticket;
    MR_TRACE_STAMP(a.trace, 0);
    pdl_trigger();
    const int nblk = blockIdx.x % a.nblocks, split = blockIdx.x / a.nblocks;
    gemv_cta<C>(a, nblk, split, blockIdx.y, red, &s_ticket, nullptr);
}

bool gemv_plan(int M, int N, int K, GemvPlan* p) {
    if (M < 1 || M > 512 || N < 8 || N > 1024 || K < 512 || K % 512 != 0) return false;
    int cfg = MR_GEMV_CFG_ROWS64;
    GemvPlan q{};
    q.cfg = cfg;
    switch (cfg) {
#define MR_PLAN_ROW(I, MT, HALF, NW, KW, KS)      \
    case I:                                       \
        q.nthr = 32 * (NW) * (KW);                \
        q.block_n = 8 * (NW);                     \
        q.rows = 16 * (MT);                       \
        q.kchunk = 32 * (KS) * (KW);              \
        break;
        MR_GEMV_CONFIGS(MR_PLAN_ROW)
#undef MR_PLAN_ROW
        default:
            return false;
    }
    if (N % q.block_n != 0 || K % q.kchunk != 0) return false;
    q.split_k = K / q.kchunk;
    q.nblocks = N / q.block_n;
    q.row_tiles = (M + q.rows - 1) / q.rows;
    if (q.row_tiles * q.nblocks > kGemvCounterSlots) return false;
    *p = q;
    return true;
}

size_t gemv_work_bytes(const GemvPlan& p, int M, int N) {
    return p.split_k > 1 ? (size_t)p.split_k * M * N * sizeof(float) : 0;
}

cudaError_t launch_router_gemv(const GemvPlan& p, const void* x, int64_t ldx, const void* w,
                               float* logits, int M, int N, int K, void* scratch,
                               cudaStream_t st) {
    GemvArgs a;
    a.x = static_cast<const uint16_t*>(x);
    a.ldx = ldx;
    a.w = static_cast<const uint16_t*>(w);
    a.logits = logits;
    a.partials = reinterpret_cast<float*>(static_cast<char*>(scratch) + kWorkOffset);
    a.counters = static_cast<unsigned*>(scratch);
    a.M = M;
    a.N = N;
    a.K = K;
    a.split_k = p.split_k;
    a.nblocks = p.nblocks;
    a.trace = static_cast<unsigned long long*>(trace_buffer());
    dim3 grid(p.nblocks * p.split_k, p.row_tiles);
    switch (p.cfg) {
#define MR_LAUNCH_ROW(I, MT, HALF, NW, KW, KS)                                              \
    case I:                                                                                 \
        return launch_kernel(router_gemv_kernel<GemvCfg<MT, HALF, NW, KW, KS>>, grid,            \
                             dim3(32 * (NW) * (KW)), 0, st, a);
        MR_GEMV_CONFIGS(MR_LAUNCH_ROW)
#undef MR_LAUNCH_ROW
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace mr
