// The one-launch route instantiated for 6 32-wide k steps per k-part
// (its own translation unit, compiled in parallel with the others; the
// kernel is in route_kernel.cuh).
#include "route_kernel.cuh"

namespace mr {

cudaError_t launch_route_cluster_spw6(const RoutePlan& p, const RouteArgs& a, cudaStream_t st) {
    return launch_route_spw<6>(p, a, st);
}

int route_timeout_flag_spw6(int clear) { return route_timeout_flag(clear); }

}  // namespace mr
