// Router GEMV alone for 64 < M <= 512 token rows and N <= 128 experts on the
// 5th-generation tensor core (tcgen05, fp32 accumulator in tensor memory).
//
// The pages' router GEMV (sglang #36557, description: split-K partial dots
// with an in-kernel fixup) at prefill-sized row counts is a small GEMM:
// D[M x N] = x[M x K] . W[N x K]^T with K = 6144.  Here one cluster of CS
// CTAs takes RPC token rows (M spread over the clusters resident at once, a
// multiple of 16) and CTA c the K slice [c*K/CS, (c+1)*K/CS):
//
//   1. The tensor memory accelerator copies the slice in stages of 64 k, one
//      128-byte swizzled row per expert or token: every weight stage before
//      the kernel waits on its predecessor (the weight is a parameter), the
//      x stages after.  Each stage lands on its own mbarrier.
//   2. One thread issues the MMAs stage by stage as the stages land:
//      D[128 expert rows x RPC tokens] += W stage . x stage^T in 16-wide
//      k-steps (weight rows past N are never written and their accumulator
//      lanes never read).
//   3. Each warp reads its quarter of the accumulator lanes (32 experts)
//      back, 16 tokens per load, and stores the partial sums to scratch as
//      [token][expert] rows of its slice (a warp's stores cover 128
//      consecutive bytes).
//   4. Split-K reduction through L2: after one cluster barrier (release /
//      acquire: every slice is in place), CTA c sums the CS slices of the
//      logits of its TOK rows of the cluster, in CTA order, and writes them.
//      (Exchanging the partials over distributed shared memory instead was
//      bound by the cluster's DSMEM fabric, about 90 bytes per cycle for all
//      16 CTAs together.)
//
// Every mbarrier wait is bounded in time and sets a device flag when it runs
// out; every CTA reaches the cluster barrier (no CTA returns before it).
#include <cuda.h>

#include "../../include/moe_route.h"
#include "cluster.cuh"
#include "common.cuh"
#include "internal.h"
#include "route_plan.h"

namespace mr {

struct TcGemvArgs {
    CUtensorMap tm_x;  // x [M rows][K] (row pitch ldx), bf16; box 64 k x rpc rows, 128-byte swizzle
    CUtensorMap tm_w;  // W [N rows][K], bf16; box 64 k x N rows, 128-byte swizzle
    float* logits;     // [M][N] fp32
    float* part;       // scratch: split-K partials [clusters][cs][rpc][N] fp32
    unsigned long long* trace;
    unsigned long long wait_ns;
    int M, N, kc, nq, nstage, rpc, tok, cs, tmem_cols, off_w;
    int flags;  // launch options (bit 1: a test stall, 16 bytes of the first x stage that never come)
};

// Set when a bounded wait of the tensor-core GEMV ran out (read by the host).
__device__ int g_tc_timeout;

// One thread: phase 0 of a local mbarrier, waited for at most limit_ns.
__device__ __forceinline__ bool tc_wait0(uint32_t bar, unsigned long long limit_ns) {
    bool ok = mbar_try_wait0(bar);
    if (!ok) {
        const unsigned long long t0 = global_ns();
        while (!(ok = mbar_try_wait0(bar)) && global_ns() - t0 < limit_ns) {
        }
        if (!ok) atomicExch(&g_tc_timeout, 1);
    }
    return ok;
}
// Thread 0 waits; the whole CTA learns the outcome.
__device__ __forceinline__ bool tc_cta_wait0(uint32_t bar, unsigned long long limit_ns, int* s_ok) {
    if (threadIdx.x == 0) *s_ok = tc_wait0(bar, limit_ns) ? 1 : 0;
    __syncthreads();
    return *s_ok != 0;
}

// Shared-memory matrix descriptor of a K-major tile in the 128-byte swizzle
// the tensor memory accelerator writes: rows of 128 bytes, 8-row groups 1024
// bytes apart (stride field), leading field unused (1), descriptor version
// bit, swizzle mode 2 (128 bytes).  A 16-wide k-step inside the 64-wide rows
// starts 32 bytes further; the tile itself is 1024-byte aligned.
__device__ __forceinline__ unsigned long long sw128_desc(uint32_t addr) {
    return (unsigned long long)((addr >> 4) & 0x3FFFu) | (1ull << 16) | ((unsigned long long)(1024 >> 4) << 32) |
           (1ull << 46) | (2ull << 61);
}
// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N >> 3 and M >> 4.
__device__ __forceinline__ uint32_t bf16_idesc(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__global__ void __launch_bounds__(kRouteThreads, 1) tc_gemv_kernel(const __grid_constant__ TcGemvArgs a) {
    extern __shared__ unsigned char dsm[];
    __shared__ __align__(8) unsigned long long s_full[kTcMaxStages];   // x stage s landed
    __shared__ __align__(8) unsigned long long s_wfull[kTcMaxStages];  // weight stage s landed
    __shared__ __align__(8) unsigned long long s_mma;                  // the CTA's MMAs done
    __shared__ int s_ok[2];
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned c = cluster_rank();
    const int cl = (int)(blockIdx.x / (unsigned)a.cs);
    const int row0 = cl * a.rpc, Mq = min(a.rpc, a.M - row0);
    const int N = a.N, tok = a.tok, rpc = a.rpc;
    const int my_rows = max(0, min(tok, Mq - (int)c * tok));
    const uint32_t base = (smem_u32(dsm) + 1023u) & ~1023u;
    const uint32_t xs = base, ws = base + (uint32_t)a.off_w;
    const uint32_t bar_mma = smem_u32(&s_mma);
    const int kslice = (int)c * a.kc;
    const uint32_t xstage = (uint32_t)rpc * 128u;
    MR_TRACE_STAMP(a.trace, 0);
    if (tid == 0) {
        for (int s = 0; s < a.nstage; ++s) {
            mbar_init(smem_u32(&s_full[s]), 1);
            mbar_init(smem_u32(&s_wfull[s]), 1);
        }
        mbar_init(bar_mma, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tma_prefetch_map(&a.tm_w);
        tma_prefetch_map(&a.tm_x);
        for (int s = 0; s < a.nstage; ++s) {
            const uint32_t full = smem_u32(&s_wfull[s]);
            mbar_expect_tx(full, (unsigned)(N * kTcStageK * 2));
            tma_load_2d(ws + (uint32_t)(s * kTcWStageBytes), &a.tm_w, kslice + s * kTcStageK, 0, full);
        }
    }
    if (warp == 0) {  // accumulator columns
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(a.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    pdl_trigger();
    pdl_wait();  // (also orders this launch's partial stores after the previous launch's reads)
    MR_TRACE_STAMP(a.trace, 8);
    if (tid == 0)
        for (int s = 0; s < a.nstage; ++s) {
            const uint32_t full = smem_u32(&s_full[s]);
            const unsigned stall = ((a.flags & 2) && s == 0) ? 16u : 0u;
            mbar_expect_tx(full, (unsigned)(rpc * kTcStageK * 2) + stall);
            tma_load_2d(xs + (uint32_t)s * xstage, &a.tm_x, kslice + s * kTcStageK, row0, full);
        }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    // ---- MMAs, stage by stage as the copies land
    if (tid == 0) {
        int fail = 0;
        const uint32_t idesc = bf16_idesc(128, rpc);
        for (int s = 0; s < a.nstage; ++s) {
            // (after a wait that ran out, the later stages are still waited
            // for, bounded, so that no copy is left in flight)
            if (!tc_wait0(smem_u32(&s_wfull[s]), a.wait_ns)) fail = 1;
            if (!tc_wait0(smem_u32(&s_full[s]), a.wait_ns)) fail = 1;
            MR_TRACE_STAMP(a.trace, 16 + s);
            if (fail) continue;
            tc_fence_after();
            const uint32_t wa = ws + (uint32_t)(s * kTcWStageBytes), xa = xs + (uint32_t)s * xstage;
#pragma unroll
            for (int j = 0; j < kTcStageK / 16; ++j) {
                const int kk = s * (kTcStageK / 16) + j;
                if (kk >= a.nq) break;
                asm volatile(
                    "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
                    "l"(sw128_desc(wa + 32u * j)), "l"(sw128_desc(xa + 32u * j)), "r"(idesc), "r"((uint32_t)(kk > 0))
                    : "memory");
            }
        }
        s_ok[1] = fail;
        // arrives once every MMA issued above has completed
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar_mma)
                     : "memory");
        MR_TRACE_STAMP(a.trace, 1);
    }
    const bool mma_ok = tc_cta_wait0(bar_mma, a.wait_ns, &s_ok[0]) && s_ok[1] == 0;
    MR_TRACE_STAMP(a.trace, 9);

    // ---- accumulator -> this CTA's slice of the partials: warp w reads
    //      lanes (experts) 32 (w % 4) .. + 31, column blocks of 16 tokens
    //      w / 4 and w / 4 + 4; for each token a warp stores 32 consecutive
    //      experts
    tc_fence_after();
    const int e = (warp & 3) * 32 + lane;
    if (mma_ok) {
        uint32_t v[2][16];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int cb = (warp >> 2) + 4 * i;
            if (cb * 16 < rpc)
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
                    "[%16];"
                    : "=r"(v[i][0]), "=r"(v[i][1]), "=r"(v[i][2]), "=r"(v[i][3]), "=r"(v[i][4]), "=r"(v[i][5]),
                      "=r"(v[i][6]), "=r"(v[i][7]), "=r"(v[i][8]), "=r"(v[i][9]), "=r"(v[i][10]), "=r"(v[i][11]),
                      "=r"(v[i][12]), "=r"(v[i][13]), "=r"(v[i][14]), "=r"(v[i][15])
                    : "r"(tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(cb * 16)));
        }
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (e < N) {
            float* slice = a.part + ((int64_t)cl * a.cs + c) * rpc * N;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int cb = (warp >> 2) + 4 * i;
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (cb * 16 + j < Mq) slice[(cb * 16 + j) * N + e] = __uint_as_float(v[i][j]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(a.tmem_cols) : "memory");
    }
    MR_TRACE_STAMP(a.trace, 10);
    // every slice of the cluster is in place (every CTA reaches this point)
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    MR_TRACE_STAMP(a.trace, 2);

    // ---- CTA c: split-K sum of the logits of its rows over the CS slices,
    //      in CTA order
    const float* rows = a.part + (int64_t)cl * a.cs * rpc * N + (int64_t)((int)c * tok) * N;
    const int plane = rpc * N;  // floats between two slices
    const int n = tid & 127;    // expert n (N <= 128) of rows tid / 128, + 4, ...
    for (int rl = tid >> 7; rl < my_rows && n < N; rl += kRouteThreads / 128) {
        const float* pp = rows + rl * N + n;
        float sum = 0.0f;
        for (int sl = 0; sl < a.cs; sl += 8) {  // cs is 8 or 16: loads first, then the adds in order
            float t8[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) t8[u] = __ldcg(pp + (sl + u) * plane);
#pragma unroll
            for (int u = 0; u < 8; ++u) sum = __fadd_rn(sum, t8[u]);
        }
        a.logits[(int64_t)(row0 + (int)c * tok + rl) * N + n] = sum;
    }
    MR_TRACE_STAMP(a.trace, 3);
}

namespace {

// cuTensorMapEncodeTiled, from the driver through the runtime's entry-point
// query (the library links only the CUDA runtime).
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
    static EncodeTiled fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        cudaGetLastError();
        return reinterpret_cast<EncodeTiled>(f);
    }();
    return fn;
}

// A 2-D bf16 tensor map over rows x cols (row pitch pitch_elems) with a box
// of 64 columns x box_rows rows in the 128-byte swizzle.
bool encode_rows(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t pitch_elems, int box_rows) {
    const EncodeTiled fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(pitch_elems * 2)};
    const cuuint32_t box[2] = {(cuuint32_t)kTcStageK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int g_prepared[64];  // per device: kernel attributes set

}  // namespace

int launch_tc_gemv(const TcGemvPlan& p, const void* x, int64_t ldx, const void* w, float* logits, int M, int N,
                   int K, void* part, cudaStream_t st, cudaError_t* err) {
    int dev = 0;
    if ((*err = cudaGetDevice(&dev)) != cudaSuccess) return MR_ERR_CUDA;
    if (dev < 0 || dev >= 64) return MR_ERR_UNSUPPORTED;
    TcGemvArgs a{};
    if (!encode_rows(&a.tm_x, x, M, K, ldx, p.rpc) || !encode_rows(&a.tm_w, w, N, K, K, N)) return MR_ERR_UNSUPPORTED;
    a.logits = logits;
    a.part = static_cast<float*>(part);
    a.trace = static_cast<unsigned long long*>(trace_buffer());
    a.wait_ns = wait_limit_ns();
    a.M = M;
    a.N = N;
    a.kc = p.kc;
    a.nq = p.nq;
    a.nstage = p.nstage;
    a.rpc = p.rpc;
    a.tok = p.tok;
    a.cs = p.cs;
    a.tmem_cols = p.tmem_cols;
    a.off_w = p.off_w;
    a.flags = launch_flags();
    if (!g_prepared[dev]) {
        if ((*err = cudaFuncSetAttribute(tc_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemMax)) !=
                cudaSuccess ||
            (*err = cudaFuncSetAttribute(tc_gemv_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) !=
                cudaSuccess)
            return MR_ERR_CUDA;
        g_prepared[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.cs * p.clusters);
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
    cudaError_t e = cudaLaunchKernelEx(&cfg, tc_gemv_kernel, a);
    if (e == cudaSuccess) e = cudaGetLastError();
    *err = e;
    return e == cudaSuccess ? MR_OK : MR_ERR_CUDA;
}

int tc_gemv_device_error(int clear) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_timeout, sizeof(int)) != cudaSuccess) return -1;
    if (clear && v) {
        const int z = 0;
        if (cudaMemcpyToSymbol(g_tc_timeout, &z, sizeof(int)) != cudaSuccess) return -1;
    }
    return v;
}

}  // namespace mr
