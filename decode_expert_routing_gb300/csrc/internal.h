// Host-side plan and launchers shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

namespace mr {

// Counter slots inside the scratch prefix (MR_SCRATCH_COUNTER_BYTES = 32 KiB).
constexpr int kCounterSlots = 8192;
constexpr int kGemvCounterSlots = 4096;   // [row_tile * nblocks + nblk]
constexpr int kFusedCounterSlot = 4096;   // fused route, several clusters: clusters done
constexpr int kSortCounterSlot = 4097;    // multi-CTA sort: completed chunks
constexpr size_t kWorkOffset = 32768;     // work area (partials or sort tables)

// Assignments one sort CTA handles.
constexpr int kSortChunk = 2048;
constexpr int kSortThreads = 256;

// One row of the per-M-bucket tiling table (the kernels are instantiated for
// exactly these rows; see gemv_configs.h).
struct GemvPlan {
    int cfg;          // index into the table
    int nthr;         // threads per CTA
    int block_n;      // experts per CTA
    int rows;         // token rows per CTA (row tile)
    int kchunk;       // K per CTA
    int split_k;      // CTAs along K
    int nblocks;      // N / block_n
    int row_tiles;    // ceil(M / rows)
};

bool gemv_plan(int M, int N, int K, GemvPlan* p);
size_t gemv_work_bytes(const GemvPlan& p, int M, int N);
size_t sort_work_bytes(int n_assign, int N);
int topk_npl(int N);  // keys per lane of the gate: 4, 8, 16 or 32

cudaError_t launch_router_gemv(const GemvPlan& p, const void* x, int64_t ldx, const void* w,
                               float* logits, int M, int N, int K, void* scratch,
                               cudaStream_t st);
cudaError_t launch_topk(const float* logits, int M, int N, int topk, int scoring,
                        const float* bias, int renormalize, int32_t* ids, float* weights,
                        cudaStream_t st);
cudaError_t launch_sort(const int32_t* ids, int M, int topk, int N, int block, int32_t* sorted,
                        int32_t* expert_ids, int32_t* ntpp, int64_t capacity, void* scratch,
                        cudaStream_t st);
cudaError_t launch_quant(const void* x, int64_t ldx, int M, int K, uint8_t* q, uint8_t* scale, bool fp4,
                         cudaStream_t st);
// One-launch parallel sort (every CTA counts every id): up to this many
// assignments, at most kPSortMaxOwn placed by one CTA.
constexpr int kPSortMaxAssign = 65536;
constexpr int kPSortMaxOwn = 2048;
constexpr int kPSortStageMax = 16384;  // ids staged in shared memory up to here (64 KiB)
struct SortArgs;
// fmt: 0 sort only, 1 MXFP8, 2 MXFP4 of x; sorted_rows: q and scale hold the
// quantised rows at the sorted positions (capacity rows) instead of token order.
cudaError_t launch_psort(const SortArgs& s, int M, int topk, const void* x, int64_t ldx, int K, uint8_t* q,
                         uint8_t* scale, int fmt, bool sorted_rows, cudaStream_t st);
cudaError_t launch_norm_apply(const void* x, int64_t ldx, const float* rstd, const void* g, int gemma, int M,
                              int K, void* xn, cudaStream_t st);
struct RoutePlan;
struct RouteArgs;
// Cluster route kernel (M <= 64): logits only (mode 0) or the whole route.
int route_cluster_size();  // 16 when the device runs 16-CTA clusters, else 8
int route_max_clusters();  // clusters of route_cluster_size() CTAs that fit on the device at once
// 1 if a bounded wait of the route kernel ran out on the current device, 0
// if not, -1 on a CUDA error; clear resets the flag.  Synchronous.
int route_device_error(int clear);
unsigned long long wait_limit_ns();
cudaError_t launch_route_cluster(const RoutePlan& p, const RouteArgs& a, cudaStream_t st);
// the instantiations for 6 and 7 k steps per k-part (kernel_route_spw6.cu,
// kernel_route_spw7.cu) and their bounded-wait flags
cudaError_t launch_route_cluster_spw6(const RoutePlan& p, const RouteArgs& a, cudaStream_t st);
cudaError_t launch_route_cluster_spw7(const RoutePlan& p, const RouteArgs& a, cudaStream_t st);
int route_timeout_flag_spw6(int clear);
int route_timeout_flag_spw7(int clear);
// Router GEMV alone above 64 rows on tcgen05 (tensor maps encoded here),
// its split-K partials in part (p.part_bytes, 16-byte aligned); returns an
// mr_status, with the CUDA error in *err on MR_ERR_CUDA.
// tc_gemv_device_error: as route_device_error, for its bounded waits.
struct TcGemvPlan;
int launch_tc_gemv(const TcGemvPlan& p, const void* x, int64_t ldx, const void* w, float* logits, int M, int N,
                   int K, void* part, cudaStream_t st, cudaError_t* err);
int tc_gemv_device_error(int clear);

// Launch options (MR_LAUNCH_* bits of mr_set_launch_flags).
int launch_flags();
// With MR_LAUNCH_CHECK_SCRATCH: MR_ERR_SCRATCH_DIRTY unless every counter of
// the scratch prefix is zero (copied to the host on st and waited for);
// MR_OK when the check is off.
int check_counters(const void* scratch, cudaStream_t st);
// Device buffer for phase stamps of tracing builds (nullptr otherwise).
void* trace_buffer();

// Launches kernel<<<grid, block, smem, st>>>(args...) through
// cudaLaunchKernelEx, allowing programmatic dependent launch when the
// MR_LAUNCH_PDL flag is set; returns the launch status.
template <class... KArgs, class... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = (launch_flags() & 1) ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Opt a kernel into more than 48 KiB of dynamic shared memory, once per
// device.
cudaError_t ensure_smem(const void* func, int bytes, int* done_per_device);

}  // namespace mr
