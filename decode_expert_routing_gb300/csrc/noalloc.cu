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
void* g_scratch_ptr[64];  // per device: device address of g_noalloc_scratch, or nullptr

// Once per device, with that device current: fetch the array's device address
// and zero its counter prefix (the split-K counters must start at zero; every
// later call leaves them at zero again).
int scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MR_ERR_CUDA;
    if (dev < 0 || dev >= 64) return MR_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MR_ERR_CUDA;
        if (cudaMemset(p, 0, MR_SCRATCH_COUNTER_BYTES) != cudaSuccess) return MR_ERR_CUDA;
        if (cudaDeviceSynchronize() != cudaSuccess) return MR_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
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
    void* scratch = nullptr;
    const int s = scratch_for_current_device(&scratch);
    if (s != MR_OK) return s;
    const cudaError_t e =
        mr::launch_router_gemv(p, x, ldx, w, logits, M, N, K, scratch, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MR_OK : MR_ERR_CUDA;
}
