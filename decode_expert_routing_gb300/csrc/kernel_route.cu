// Host side of the one-launch route (the kernel and its launch are in
// route_kernel.cuh): the device's cluster support, the dispatch to the
// instantiation of the launch's step count, and the bounded-wait flags.
// This unit instantiates the run-time step count; kernel_route_spw6.cu and
// kernel_route_spw7.cu the common ones.
#include "route_kernel.cuh"

namespace mr {

int route_device_error(int clear) {
    const int v0 = route_timeout_flag(clear), v6 = route_timeout_flag_spw6(clear), v7 = route_timeout_flag_spw7(clear);
    if (v0 < 0 || v6 < 0 || v7 < 0) return -1;
    return v0 | v6 | v7;
}

static int g_cluster16[64];     // per device: 0 unknown, 1 usable, -1 not

int route_cluster_size() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 8;
    if (g_cluster16[dev] == 0) {
        cudaError_t e = prepare<false, false, kKindSoftmax, false, 0>(dev);
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
            e = cudaOccupancyMaxActiveClusters(&n, route_cluster_kernel<false, false, kKindSoftmax, false, 0>, &cfg);
        }
        g_cluster16[dev] = (e == cudaSuccess && n >= 1) ? 1 : -1;
        cudaGetLastError();  // a refused query leaves no sticky error
    }
    return g_cluster16[dev] > 0 ? 16 : 8;
}

static int g_max_clusters[64];  // per device: co-resident clusters of the mma.sync kernel (0: unknown)

int route_max_clusters() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (g_max_clusters[dev] == 0) {
        const int cs = route_cluster_size();
        int n = 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cs);
        cfg.blockDim = dim3(kRouteThreads);
        cfg.dynamicSmemBytes = kRouteSmemMax;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = cs;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, route_cluster_kernel<false, false, kKindSoftmax, false, 0>, &cfg);
        g_max_clusters[dev] = (e == cudaSuccess && n >= 1) ? n : 1;
        cudaGetLastError();
    }
    return g_max_clusters[dev];
}

cudaError_t launch_route_cluster(const RoutePlan& p, const RouteArgs& a, cudaStream_t st) {
    // the step count of the route's clusters and of the shared expert's, when
    // the launch has both they must agree to take a fixed-count instantiation
    const int rs = p.clusters > 0 ? a.spw : 0, ss = p.sh_clusters > 0 ? a.sh_spw : 0;
    const int spw = rs == 0 ? ss : (ss == 0 || ss == rs ? rs : 0);
    if (spw == 6) return launch_route_cluster_spw6(p, a, st);
    if (spw == 7) return launch_route_cluster_spw7(p, a, st);
    return launch_route_spw<0>(p, a, st);
}

}  // namespace mr
