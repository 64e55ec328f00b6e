// Router GEMV whose split-K scratch lives in this library's own device
// memory, for callers that cannot call cudaMalloc (see mr_router_gemv_noalloc
// in moe_route.h).  Nothing here allocates: the scratch is a file-scope
// __device__ array that the CUDA runtime places when the module loads.
#include <stdint.h>

#include <mutex>

#include "../../include/moe_route.h"
#include "internal.h"

namespace {

// Counter prefix + split-K partials of every call of mr_router_gemv_noalloc.
// Every GPU that loads this library holds these bytes until the process
// exits.  Device code could also name the array; host code must use the
// address that cudaGetSymbolAddress returns (the name is a host stand-in).
static __device__ __align__(256) unsigned char g_noalloc_scratch[MR_NOALLOC_SCRATCH_BYTES];

std::mutex g_setup_mutex;

// Per device: the array's device address and the context it was looked up
// in, as of the last set-up.
struct Placement {
    void* ptr;
    void* ctx;
};
Placement g_placement[64];

// The calling thread's current CUDA context (a driver handle), or nullptr if
// the driver entry point is unavailable.  A context that is destroyed and
// created again (cudaDeviceReset) loads this module again, possibly at
// another address and with its contents undefined.
void* current_context() {
    using GetCtx = int (*)(void**);
    static GetCtx fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<GetCtx>(f);
    }();
    void* ctx = nullptr;
    if (fn == nullptr || fn(&ctx) != 0) return nullptr;
    return ctx;
}

// The array's device address for the current device, looked up on every
// call (host code only sees a stand-in under its name).  The first call in a
// context, or one that finds the array at a new address, zeroes the counter
// prefix on the call's stream (the split-K counters must start at zero;
// every later call leaves them at zero again).
int scratch_for_current_device(cudaStream_t st, void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MR_ERR_CUDA;
    if (dev < 0 || dev >= 64) return MR_ERR_UNSUPPORTED;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MR_ERR_CUDA;
    void* ctx = current_context();
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    Placement& pl = g_placement[dev];
    if (pl.ptr != p || pl.ctx != ctx || ctx == nullptr) {  // (no context handle: zero on every call)
        if (cudaMemsetAsync(p, 0, MR_SCRATCH_COUNTER_BYTES, st) != cudaSuccess) return MR_ERR_CUDA;
        pl.ptr = p;
        pl.ctx = ctx;
    }
    *out = p;
    return MR_OK;
}

}  // namespace

extern "C" int mr_router_gemv_noalloc(const void* x, int64_t ldx, const void* w, float* logits, int M,
                                      int N, int K, void* stream) {
    if (x == nullptr || w == nullptr || logits == nullptr) return MR_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(w) & 15) ||
        (reinterpret_cast<uintptr_t>(logits) & 7))
        return MR_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1 || ldx < K || ldx % 8 != 0) return MR_ERR_INVALID_ARG;
    mr::GemvPlan p;
    if (!mr::gemv_plan(M, N, K, &p)) return MR_ERR_UNSUPPORTED;
    // the built-in scratch has a fixed size: larger problems are refused
    if (mr::kWorkOffset + mr::gemv_work_bytes(p, M, N) > (size_t)MR_NOALLOC_SCRATCH_BYTES)
        return MR_ERR_UNSUPPORTED;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    void* scratch = nullptr;
    int s = scratch_for_current_device(st, &scratch);
    if (s != MR_OK) return s;
    if ((s = mr::check_counters(scratch, st)) != MR_OK) return s;
    const cudaError_t e = mr::launch_router_gemv(p, x, ldx, w, logits, M, N, K, scratch, st);
    return e == cudaSuccess ? MR_OK : MR_ERR_CUDA;
}
