// C ABI entry points: host-side validation, then one launcher call each.
// Nothing here allocates device memory.
#include <stdint.h>

#include <atomic>

#include "../../include/moe_route.h"
#include "internal.h"
#include "route_plan.h"
#include "sort.cuh"

namespace {

using mr::GemvPlan;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

thread_local int g_last_cuda_error = 0;  // behind this thread's last MR_ERR_CUDA

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return MR_OK;
    g_last_cuda_error = (int)e;
    return MR_ERR_CUDA;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

// Common checks of an x operand.
int check_x(const void* x, int64_t ldx, int M, int K) {
    if (x == nullptr || !aligned(x, 16)) return MR_ERR_INVALID_ARG;
    if (M < 1 || K < 1 || ldx < K || ldx % 8 != 0) return MR_ERR_INVALID_ARG;
    return MR_OK;
}

int check_gate_args(int M, int N, int topk, int scoring) {
    if (M < 1 || N < 1) return MR_ERR_INVALID_ARG;
    if (scoring != MR_SCORE_SOFTMAX && scoring != MR_SCORE_SIGMOID) return MR_ERR_INVALID_ARG;
    if (topk < 1 || topk > N) return MR_ERR_INVALID_ARG;
    if (N > MR_MAX_EXPERTS || topk > MR_MAX_TOPK) return MR_ERR_UNSUPPORTED;
    return MR_OK;
}

int check_sort_args(int M, int topk, int N, int block, int64_t capacity) {
    if (M < 1 || topk < 1 || N < 1 || block < 1) return MR_ERR_INVALID_ARG;
    if (N > MR_MAX_EXPERTS || topk > MR_MAX_TOPK || block > 1024) return MR_ERR_UNSUPPORTED;
    const int64_t need = mr_sort_capacity(M, topk, N, block);
    if (need < 0) return MR_ERR_UNSUPPORTED;
    if (capacity < need) return MR_ERR_INVALID_ARG;
    return MR_OK;
}

std::atomic<int> g_launch_flags{0};
std::atomic<unsigned long long> g_wait_ns{1000000000ull};
std::atomic<void*> g_trace{nullptr};

}  // namespace

namespace mr {
int launch_flags() { return g_launch_flags.load(std::memory_order_relaxed); }
}  // namespace mr
namespace {
bool allow_tc() { return (mr::launch_flags() & MR_LAUNCH_LEGACY_MMA) == 0; }
}  // namespace
namespace mr {
int check_counters(const void* scratch, cudaStream_t st) {
    if ((mr::launch_flags() & MR_LAUNCH_CHECK_SCRATCH) == 0) return MR_OK;
    static thread_local unsigned host[MR_SCRATCH_COUNTER_BYTES / sizeof(unsigned)];
    if (cudaMemcpyAsync(host, scratch, MR_SCRATCH_COUNTER_BYTES, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return MR_ERR_CUDA;
    for (unsigned v : host)
        if (v != 0u) return MR_ERR_SCRATCH_DIRTY;
    return MR_OK;
}
}  // namespace mr
namespace {
using mr::check_counters;
}  // namespace
namespace mr {
unsigned long long wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
void* trace_buffer() { return g_trace.load(std::memory_order_relaxed); }
}  // namespace mr

extern "C" {

int mr_set_launch_flags(int flags) {
    if (flags & ~(MR_LAUNCH_PDL | MR_LAUNCH_TEST_STALL | MR_LAUNCH_LEGACY_MMA | MR_LAUNCH_TEST_SLOW_SIGMOID |
                  MR_LAUNCH_CHECK_SCRATCH))
        return MR_ERR_INVALID_ARG;
    g_launch_flags.store(flags, std::memory_order_relaxed);
    return MR_OK;
}

int mr_get_launch_flags(void) { return g_launch_flags.load(std::memory_order_relaxed); }

int mr_set_wait_limit_ns(uint64_t ns) {
    if (ns < 1000ull || ns > 60000000000ull) return MR_ERR_INVALID_ARG;
    g_wait_ns.store(ns, std::memory_order_relaxed);
    return MR_OK;
}

int mr_device_error(int clear) {
    const int v = mr::route_device_error(clear), t = mr::tc_gemv_device_error(clear);
    return (v < 0 || t < 0) ? MR_ERR_CUDA : (v || t) ? MR_ERR_TIMEOUT : MR_OK;
}

#ifdef MR_TRACE
// Tracing builds only: device buffer of gridDim * 256 u64 stamps for the next
// launches (nullptr stops tracing).
int mr_trace_set_buffer(void* device_buffer) {
    g_trace.store(device_buffer, std::memory_order_relaxed);
    return MR_OK;
}
#endif

const char* mr_status_string(int status) {
    switch (status) {
        case MR_OK: return "MR_OK";
        case MR_ERR_UNSUPPORTED: return "MR_ERR_UNSUPPORTED: shape or layout outside the kernels' cover";
        case MR_ERR_INVALID_ARG: return "MR_ERR_INVALID_ARG: null or misaligned pointer, or bad size";
        case MR_ERR_SCRATCH_TOO_SMALL: return "MR_ERR_SCRATCH_TOO_SMALL: scratch_bytes below what the call needs";
        case MR_ERR_CUDA: return "MR_ERR_CUDA: the CUDA runtime reported an error";
        case MR_ERR_TIMEOUT: return "MR_ERR_TIMEOUT: a kernel's bounded wait for data from other CTAs ran out";
        case MR_ERR_SCRATCH_DIRTY:
            return "MR_ERR_SCRATCH_DIRTY: scratch counters not zero before the launch (never zeroed, or in use)";
        default: return "unknown mr_status";
    }
}

int mr_abi_version(void) { return MR_ABI_VERSION; }

int mr_last_cuda_error(void) { return g_last_cuda_error; }

int mr_router_gemv_supported(int M, int N, int K, int64_t ldx) {
    if (ldx < K || ldx % 8 != 0 || K % MR_GEMV_K_MULTIPLE != 0) return 0;
    mr::RoutePlan rp;
    mr::TcGemvPlan tp;
    if (mr::route_plan(M, N, K, 1, 0, 16, &rp) || mr::tc_gemv_plan(M, N, K, 16, 1, &tp)) return 1;
    if (M <= mr::kRouteMaxM) return 0;
    GemvPlan p;
    return mr::gemv_plan(M, N, K, &p) ? 1 : 0;
}

int64_t mr_sort_capacity(int M, int topk, int N, int block) {
    if (M < 1 || topk < 1 || N < 1 || block < 1) return -1;
    const int64_t mk = (int64_t)M * topk;
    const int64_t used = mk < N ? mk : N;
    const int64_t cap = (mk + used * (block - 1) + block - 1) / block * block;
    if (cap >= ((int64_t)1 << 31)) return -1;  // positions are stored as int32
    return cap;
}

size_t mr_scratch_bytes(int M_max, int N, int K, int topk) {
    if (M_max < 1 || N < 1 || K < 1 || topk < 1) return 0;
    size_t work = 0;
    const int Mg = M_max < MR_MAX_GEMV_ROWS ? M_max : MR_MAX_GEMV_ROWS;
    for (int M = mr::kRouteMaxM + 1; M <= Mg; ++M) {
        GemvPlan p;
        if (mr::gemv_plan(M, N, K, &p)) {
            const size_t b = mr::gemv_work_bytes(p, M, N);
            if (b > work) work = b;
        }
        mr::TcGemvPlan tp;  // the tensor-core GEMV's partials (a bound over every resident-cluster count)
        if (mr::tc_gemv_plan(M, N, K, 16, 1, &tp)) {
            const size_t b = (size_t)mr::tc_gemv_part_bound(M, N);
            if (b > work) work = b;
        }
    }
    if (M_max > mr::kRouteRowsPerCluster) {  // fused route over several clusters: every token's ids
        const int Mf = M_max < mr::kRouteMaxM ? M_max : mr::kRouteMaxM;
        const size_t b = (size_t)Mf * topk * 4;
        if (b > work) work = b;
    }
    if (N >= mr::kRouteSplitMinN) {  // fused route over expert groups (one token group): their candidates
        const int Mf = M_max < mr::kRouteRowsPerCluster ? M_max : mr::kRouteRowsPerCluster;
        const size_t b = (size_t)Mf * mr::kRouteMaxGroups * topk * 12;
        if (b > work) work = b;
    }
    const int64_t n_assign = (int64_t)M_max * topk;
    if (n_assign > mr::kPSortMaxAssign && n_assign < ((int64_t)1 << 30)) {
        const size_t b = mr::sort_work_bytes((int)n_assign, N);
        if (b > work) work = b;
    }
    return mr::kWorkOffset + ((work + 255) / 256) * 256;
}

int mr_scratch_reset(void* scratch, size_t scratch_bytes, void* stream) {
    if (scratch == nullptr || scratch_bytes < MR_SCRATCH_COUNTER_BYTES) return MR_ERR_INVALID_ARG;
    return cuda_status(cudaMemsetAsync(scratch, 0, scratch_bytes, as_stream(stream)));
}

// Fills the cluster route arguments shared by the GEMV-only and full modes.
static mr::RouteArgs route_args(const mr::RoutePlan& p, const void* x, int64_t ldx, const void* w, int M,
                                int N, int K, int mode) {
    mr::RouteArgs a{};
    a.x = static_cast<const uint16_t*>(x);
    a.ldx = ldx;
    a.w = static_cast<const uint16_t*>(w);
    a.M = M;
    a.N = p.nl;   // experts of one cluster (all of them unless split into groups)
    a.ldn = N;
    a.ng = p.ng;
    a.off_merge = p.off_merge;
    a.K = K;
    a.mode = mode;
    a.cs = p.cs;
    a.cs_shift = mr::ilog2_exact(p.cs);
    a.rpc = p.rpc;
    a.clusters = p.clusters;
    a.kc = p.kc;
    a.spw = p.spw;
    a.wpt = p.wpt;
    a.units = p.units;
    a.tok = p.tok;
    a.xpitch = p.xpitch;
    a.off_x = p.off_x;
    a.off_recv = p.off_recv;
    a.off_row = p.off_row;
    a.off_key = p.off_key;
    a.off_cand = p.off_cand;
    a.off_ids = p.off_ids;
    a.off_mask = p.off_mask;
    a.off_start = p.off_start;
    a.off_kred = p.off_kred;
    a.tok_shift = mr::ilog2_exact(p.tok);
    a.wpt_shift = mr::ilog2_exact(p.wpt);
    a.mag_n = mr::div_magic(p.nl);
    a.mag_vpr = mr::div_magic(p.kc / 8);
    a.mag_n4 = mr::div_magic(N / 4 > 0 ? N / 4 : 1);
    a.nslots = p.nslots;
    a.trace = static_cast<unsigned long long*>(mr::trace_buffer());
    a.flags = mr::launch_flags();
    a.wait_ns = mr::wait_limit_ns();
    return a;
}

int mr_router_gemv(const void* x, int64_t ldx, const void* w, float* logits, int M, int N, int K,
                   void* scratch, size_t scratch_bytes, void* stream) {
    int s = check_x(x, ldx, M, K);
    if (s != MR_OK) return s;
    if (w == nullptr || !aligned(w, 16) || logits == nullptr || !aligned(logits, 8) || N < 1)
        return MR_ERR_INVALID_ARG;
    if (K % MR_GEMV_K_MULTIPLE != 0) return MR_ERR_UNSUPPORTED;
    if (M > mr::kRouteMaxM && allow_tc()) {  // above 64 rows: tcgen05 when its plan and the scratch fit
        mr::TcGemvPlan tp;
        if (mr::tc_gemv_plan(M, N, K, mr::route_cluster_size(), mr::route_max_clusters(), &tp) &&
            scratch != nullptr && aligned(scratch, 256) &&
            scratch_bytes >= mr::kWorkOffset + (size_t)tp.part_bytes) {
            cudaError_t e = cudaSuccess;
            void* part = static_cast<unsigned char*>(scratch) + mr::kWorkOffset;
            const int st = mr::launch_tc_gemv(tp, x, ldx, w, logits, M, N, K, part, as_stream(stream), &e);
            return st == MR_ERR_CUDA ? cuda_status(e) : st;
        }
    }
    {   // the cluster kernel (no scratch) whenever its plan fits; above 64 rows
        // the split-K GEMV with last-arriver fixup takes the rest
        mr::RoutePlan rp;
        if (mr::route_plan(M, N, K, 1, 0, mr::route_cluster_size(), &rp, mr::route_max_clusters())) {
            mr::RouteArgs a = route_args(rp, x, ldx, w, M, N, K, 0);
            a.logits = logits;
            return cuda_status(mr::launch_route_cluster(rp, a, as_stream(stream)));
        }
        if (M <= mr::kRouteMaxM) return MR_ERR_UNSUPPORTED;
    }
    if (scratch == nullptr || !aligned(scratch, 256)) return MR_ERR_INVALID_ARG;
    GemvPlan p;
    if (!mr::gemv_plan(M, N, K, &p)) return MR_ERR_UNSUPPORTED;
    if (scratch_bytes < mr::kWorkOffset + mr::gemv_work_bytes(p, M, N)) return MR_ERR_SCRATCH_TOO_SMALL;
    if ((s = check_counters(scratch, as_stream(stream))) != MR_OK) return s;
    return cuda_status(mr::launch_router_gemv(p, x, ldx, w, logits, M, N, K, scratch, as_stream(stream)));
}

int mr_route_topk(const float* logits, int M, int N, int topk, int scoring, const float* sel_bias,
                  int renormalize, int32_t* topk_ids, float* topk_weights, void* stream) {
    int s = check_gate_args(M, N, topk, scoring);
    if (s != MR_OK) return s;
    if (logits == nullptr || !aligned(logits, 4) || topk_ids == nullptr || !aligned(topk_ids, 4) ||
        topk_weights == nullptr || !aligned(topk_weights, 4) || (sel_bias && !aligned(sel_bias, 4)))
        return MR_ERR_INVALID_ARG;
    return cuda_status(mr::launch_topk(logits, M, N, topk, scoring, scoring == MR_SCORE_SIGMOID ? sel_bias : nullptr,
                                       renormalize ? 1 : 0, topk_ids, topk_weights, as_stream(stream)));
}

int mr_moe_sort(const int32_t* topk_ids, int M, int topk, int N, int block, int32_t* sorted_token_ids,
                int32_t* expert_ids, int32_t* num_tokens_post_padded, int64_t capacity, void* scratch,
                size_t scratch_bytes, void* stream) {
    int s = check_sort_args(M, topk, N, block, capacity);
    if (s != MR_OK) return s;
    if (topk_ids == nullptr || !aligned(topk_ids, 4) || sorted_token_ids == nullptr ||
        !aligned(sorted_token_ids, 4) || expert_ids == nullptr || !aligned(expert_ids, 4) ||
        num_tokens_post_padded == nullptr || !aligned(num_tokens_post_padded, 4))
        return MR_ERR_INVALID_ARG;
    const int64_t n_assign = (int64_t)M * topk;
    if (n_assign > mr::kPSortMaxAssign) {
        if (n_assign >= ((int64_t)1 << 30)) return MR_ERR_UNSUPPORTED;
        if (scratch == nullptr || !aligned(scratch, 256)) return MR_ERR_INVALID_ARG;
        if (scratch_bytes < mr::kWorkOffset + mr::sort_work_bytes((int)n_assign, N))
            return MR_ERR_SCRATCH_TOO_SMALL;
        if ((s = check_counters(scratch, as_stream(stream))) != MR_OK) return s;
    }
    return cuda_status(mr::launch_sort(topk_ids, M, topk, N, block, sorted_token_ids, expert_ids,
                                       num_tokens_post_padded, capacity, scratch, as_stream(stream)));
}

int mr_moe_sort_quant(const int32_t* topk_ids, int M, int topk, int N, int block, const void* x, int64_t ldx,
                      int K, int quant_format, int32_t* sorted_token_ids, int32_t* expert_ids,
                      int32_t* num_tokens_post_padded, int64_t capacity, uint8_t* q, uint8_t* scale, void* stream) {
    int s = check_sort_args(M, topk, N, block, capacity);
    if (s != MR_OK) return s;
    if ((s = check_x(x, ldx, M, K)) != MR_OK) return s;
    if (topk_ids == nullptr || !aligned(topk_ids, 4) || sorted_token_ids == nullptr ||
        !aligned(sorted_token_ids, 4) || expert_ids == nullptr || !aligned(expert_ids, 4) ||
        num_tokens_post_padded == nullptr || !aligned(num_tokens_post_padded, 4))
        return MR_ERR_INVALID_ARG;
    const int fmt = quant_format & ~MR_QUANT_SORTED_ROWS;
    const bool sorted_rows = (quant_format & MR_QUANT_SORTED_ROWS) != 0;
    if (fmt != MR_QUANT_MXFP8 && fmt != MR_QUANT_MXFP4) return MR_ERR_INVALID_ARG;
    if (q == nullptr || !aligned(q, 8) || scale == nullptr) return MR_ERR_INVALID_ARG;
    if (K % 32 != 0 || (int64_t)M * topk > MR_SORT_QUANT_MAX_ASSIGN) return MR_ERR_UNSUPPORTED;
    const mr::SortArgs a{topk_ids, M * topk, N, block, sorted_token_ids, expert_ids, num_tokens_post_padded, capacity};
    return cuda_status(mr::launch_psort(a, M, topk, x, ldx, K, q, scale, fmt == MR_QUANT_MXFP4 ? 2 : 1, sorted_rows,
                                        as_stream(stream)));
}

int mr_mxfp8_quant(const void* x, int64_t ldx, int M, int K, uint8_t* q, uint8_t* scale, void* stream) {
    int s = check_x(x, ldx, M, K);
    if (s != MR_OK) return s;
    if (K % 32 != 0) return MR_ERR_UNSUPPORTED;
    if (q == nullptr || !aligned(q, 8) || scale == nullptr) return MR_ERR_INVALID_ARG;
    return cuda_status(mr::launch_quant(x, ldx, M, K, q, scale, false, as_stream(stream)));
}

int mr_mxfp4_quant(const void* x, int64_t ldx, int M, int K, uint8_t* q, uint8_t* scale, void* stream) {
    int s = check_x(x, ldx, M, K);
    if (s != MR_OK) return s;
    if (K % 32 != 0) return MR_ERR_UNSUPPORTED;
    if (q == nullptr || !aligned(q, 4) || scale == nullptr) return MR_ERR_INVALID_ARG;
    return cuda_status(mr::launch_quant(x, ldx, M, K, q, scale, true, as_stream(stream)));
}

}  // extern "C"

static int check_norm(const float* rstd, const void* norm_w, int norm_kind);

// Validates the shared expert's arguments and adds its clusters to the
// launch: a's sh_* fields, rp's cluster count and shared memory.
static int shared_args(const uint8_t* w13, const uint8_t* w13_scale, int I, void* act, int M, int K, int cs,
                       mr::RouteArgs* a, mr::RoutePlan* rp) {
    if (w13 == nullptr || !aligned(w13, 16) || w13_scale == nullptr || act == nullptr || !aligned(act, 4) || I < 1)
        return MR_ERR_INVALID_ARG;
    mr::SharedPlan sp;
    const int fit = mr::route_max_clusters() - rp->clusters;
    if (!mr::shared_plan(M, K, I, cs, &sp, fit > 1 ? fit : 1)) return MR_ERR_UNSUPPORTED;
    a->sh_w = w13;
    a->sh_scale = w13_scale;
    a->sh_out = static_cast<uint16_t*>(act);
    a->sh_I = I;
    a->sh_clusters = sp.clusters;
    a->sh_pairs = sp.pairs;
    a->sh_wpt = sp.wpt;
    a->sh_spw = sp.spw;
    a->sh_units = sp.units;
    a->sh_nslots = sp.nslots;
    a->sh_off_x = sp.off_x;
    a->sh_off_recv = sp.off_recv;
    a->sh_off_w = sp.off_w;
    a->sh_off_s = sp.off_s;
    a->sh_spitch = sp.spitch;
    rp->sh_clusters = sp.clusters;
    if (sp.smem > rp->smem) rp->smem = sp.smem;
    return MR_OK;
}

// The one-launch route.  p->rstd != nullptr puts the router input on the
// norm's scale (residual rows x rstd x norm weight, rounded to bf16 in the
// kernel); p->quant_format picks the stage-1 activation format.
static int route_impl(const mr_route_params* p, void* stream) {
    if (p == nullptr) return MR_ERR_INVALID_ARG;
    const int M = p->M, N = p->N, K = p->K, topk = p->topk, scoring = p->scoring, block = p->block;
    int s = check_x(p->x, p->ldx, M, K);
    if (s != MR_OK) return s;
    if ((s = check_gate_args(M, N, topk, scoring)) != MR_OK) return s;
    if ((s = check_sort_args(M, topk, N, block, p->capacity)) != MR_OK) return s;
    if (p->rstd != nullptr && (s = check_norm(p->rstd, p->norm_weight, p->norm_kind)) != MR_OK) return s;
    if (M > MR_MAX_FUSED_ROWS || K % MR_GEMV_K_MULTIPLE != 0) return MR_ERR_UNSUPPORTED;
    if (p->w == nullptr || !aligned(p->w, 16) || p->logits == nullptr || !aligned(p->logits, 8) ||
        p->topk_ids == nullptr || !aligned(p->topk_ids, 4) || p->topk_weights == nullptr ||
        !aligned(p->topk_weights, 4) || p->sorted_token_ids == nullptr || !aligned(p->sorted_token_ids, 4) ||
        p->expert_ids == nullptr || !aligned(p->expert_ids, 4) || p->num_tokens_post_padded == nullptr ||
        !aligned(p->num_tokens_post_padded, 4) || (p->sel_bias && !aligned(p->sel_bias, 4)))
        return MR_ERR_INVALID_ARG;
    const int qf = p->quant_format;
    if (qf != MR_QUANT_NONE && qf != MR_QUANT_MXFP8 && qf != MR_QUANT_MXFP4) return MR_ERR_INVALID_ARG;
    if (qf != MR_QUANT_NONE && (p->q == nullptr || !aligned(p->q, 8) || p->scale == nullptr))
        return MR_ERR_INVALID_ARG;
    mr::RoutePlan rp;
    const int cs = mr::route_cluster_size();
    // expert groups need scratch for their candidates: without it (or with
    // too little) the route runs its experts in one cluster per 16 tokens
    const bool have_scratch = p->scratch != nullptr && aligned(p->scratch, 256);
    if (!mr::route_plan(M, N, K, topk, 1, cs, &rp, have_scratch ? mr::route_max_clusters() : 1))
        return MR_ERR_UNSUPPORTED;
    if (rp.ng > 1 && p->scratch_bytes < mr::kWorkOffset + (size_t)M * rp.ng * topk * 12 &&
        !mr::route_plan(M, N, K, topk, 1, cs, &rp, 1))
        return MR_ERR_UNSUPPORTED;
    mr::RouteArgs a = route_args(rp, p->x, p->ldx, p->w, M, N, K, 1);
    if (rp.clusters > 1) {  // the clusters meet in scratch: a ticket and every token's ids
        if (!have_scratch) return MR_ERR_INVALID_ARG;
        if (p->scratch_bytes < mr::kWorkOffset + (size_t)M * topk * 4) return MR_ERR_SCRATCH_TOO_SMALL;
        a.counter = static_cast<unsigned*>(p->scratch) + mr::kFusedCounterSlot;
        a.ids_scratch = reinterpret_cast<int32_t*>(static_cast<char*>(p->scratch) + mr::kWorkOffset);
    }
    if (rp.ng > 1) {  // each cluster's collector publishes its group candidates and takes a ticket
        char* work = static_cast<char*>(p->scratch) + mr::kWorkOffset;
        a.cand_key = reinterpret_cast<unsigned long long*>(work);
        a.cand_val = reinterpret_cast<float*>(work + (size_t)M * rp.ng * topk * 8);
    }
    if ((rp.clusters > 1 || rp.ng > 1) && (s = check_counters(p->scratch, as_stream(stream))) != MR_OK) return s;
    a.bias = scoring == MR_SCORE_SIGMOID ? p->sel_bias : nullptr;
    a.logits = p->logits;
    a.ids = p->topk_ids;
    a.weights = p->topk_weights;
    a.sorted = p->sorted_token_ids;
    a.expert_ids = p->expert_ids;
    a.ntpp = p->num_tokens_post_padded;
    a.capacity = p->capacity;
    a.q = qf == MR_QUANT_NONE ? nullptr : p->q;
    a.scale = qf == MR_QUANT_NONE ? nullptr : p->scale;
    a.quant_fp4 = qf == MR_QUANT_MXFP4 ? 1 : 0;
    a.topk = topk;
    {  // gate threshold lane groups: the largest power of two <= 32 threads
       // leaving at least topk groups that hold experts (thread t: experts t
       // and t + 512)
        const int lanes = rp.nl < 512 ? rp.nl : 512;
        int gsh = 5;
        while (gsh > 0 && (lanes + (1 << gsh) - 1) >> gsh < topk) --gsh;
        a.gs_shift = gsh;
    }
    a.block = block;
    a.mag_k = mr::div_magic(topk);
    a.mag_block = mr::div_magic(block);
    a.scoring = scoring;
    a.renormalize = p->renormalize ? 1 : 0;
    a.rstd = p->rstd;
    a.norm_w = static_cast<const uint16_t*>(p->norm_weight);
    a.norm_gemma = p->norm_kind == MR_NORM_GEMMA ? 1 : 0;
    if (p->shared_w13 != nullptr) {  // the shared expert's clusters join the launch
        if ((s = shared_args(p->shared_w13, p->shared_w13_scale, p->shared_inter, p->shared_act, M, K, cs, &a,
                             &rp)) != MR_OK)
            return s;
    }
    return cuda_status(mr::launch_route_cluster(rp, a, as_stream(stream)));
}

static int check_norm(const float* rstd, const void* norm_w, int norm_kind) {
    if (rstd == nullptr || !aligned(rstd, 4) || norm_w == nullptr || !aligned(norm_w, 16)) return MR_ERR_INVALID_ARG;
    if (norm_kind != MR_NORM_RMS && norm_kind != MR_NORM_GEMMA) return MR_ERR_INVALID_ARG;
    return MR_OK;
}

static mr_route_params fill_params(const void* x, int64_t ldx, const void* w, int M, int N, int K, int topk,
                                   int scoring, const float* sel_bias, int renormalize, int block, float* logits,
                                   int32_t* topk_ids, float* topk_weights, int32_t* sorted_token_ids,
                                   int32_t* expert_ids, int32_t* num_tokens_post_padded, int64_t capacity,
                                   uint8_t* q, uint8_t* scale, void* scratch, size_t scratch_bytes) {
    mr_route_params p{};
    p.x = x;
    p.ldx = ldx;
    p.w = w;
    p.M = M;
    p.N = N;
    p.K = K;
    p.topk = topk;
    p.scoring = scoring;
    p.sel_bias = sel_bias;
    p.renormalize = renormalize;
    p.block = block;
    p.logits = logits;
    p.topk_ids = topk_ids;
    p.topk_weights = topk_weights;
    p.sorted_token_ids = sorted_token_ids;
    p.expert_ids = expert_ids;
    p.num_tokens_post_padded = num_tokens_post_padded;
    p.capacity = capacity;
    p.q = q;
    p.scale = scale;
    p.quant_format = (q == nullptr && scale == nullptr) ? MR_QUANT_NONE : MR_QUANT_MXFP8;
    p.scratch = scratch;
    p.scratch_bytes = scratch_bytes;
    return p;
}

extern "C" {

int mr_moe_route(const mr_route_params* p, void* stream) { return route_impl(p, stream); }

int mr_moe_route_sort_quant(const void* x, int64_t ldx, const void* w, int M, int N, int K, int topk,
                            int scoring, const float* sel_bias, int renormalize, int block,
                            float* logits, int32_t* topk_ids, float* topk_weights,
                            int32_t* sorted_token_ids, int32_t* expert_ids,
                            int32_t* num_tokens_post_padded, int64_t capacity, uint8_t* q,
                            uint8_t* scale, void* scratch, size_t scratch_bytes, void* stream) {
    if ((q == nullptr) != (scale == nullptr)) return MR_ERR_INVALID_ARG;
    const mr_route_params p = fill_params(x, ldx, w, M, N, K, topk, scoring, sel_bias, renormalize, block, logits,
                                          topk_ids, topk_weights, sorted_token_ids, expert_ids,
                                          num_tokens_post_padded, capacity, q, scale, scratch, scratch_bytes);
    return route_impl(&p, stream);
}

int mr_moe_route_sort_quant_norm(const void* sres, int64_t ldx, const float* rstd, const void* norm_weight,
                                 int norm_kind, const void* w, int M, int N, int K, int topk, int scoring,
                                 const float* sel_bias, int renormalize, int block, float* logits,
                                 int32_t* topk_ids, float* topk_weights, int32_t* sorted_token_ids,
                                 int32_t* expert_ids, int32_t* num_tokens_post_padded, int64_t capacity,
                                 uint8_t* q, uint8_t* scale, void* scratch, size_t scratch_bytes, void* stream) {
    const int s = check_norm(rstd, norm_weight, norm_kind);
    if (s != MR_OK) return s;
    if ((q == nullptr) != (scale == nullptr)) return MR_ERR_INVALID_ARG;
    mr_route_params p = fill_params(sres, ldx, w, M, N, K, topk, scoring, sel_bias, renormalize, block, logits,
                                    topk_ids, topk_weights, sorted_token_ids, expert_ids, num_tokens_post_padded,
                                    capacity, q, scale, scratch, scratch_bytes);
    p.rstd = rstd;
    p.norm_weight = norm_weight;
    p.norm_kind = norm_kind;
    return route_impl(&p, stream);
}

int mr_norm_apply(const void* sres, int64_t ldx, const float* rstd, const void* norm_weight, int norm_kind, int M,
                  int K, void* xn, void* stream) {
    int s = check_x(sres, ldx, M, K);
    if (s != MR_OK) return s;
    if ((s = check_norm(rstd, norm_weight, norm_kind)) != MR_OK) return s;
    if (K % 8 != 0) return MR_ERR_UNSUPPORTED;
    if (xn == nullptr || !aligned(xn, 16)) return MR_ERR_INVALID_ARG;
    return cuda_status(mr::launch_norm_apply(sres, ldx, rstd, norm_weight, norm_kind == MR_NORM_GEMMA ? 1 : 0, M,
                                             K, xn, as_stream(stream)));
}

int mr_shared_gate_up(const void* x, int64_t ldx, const uint8_t* w13, const uint8_t* w13_scale, int M, int K,
                      int I, void* act, void* stream) {
    int s = check_x(x, ldx, M, K);
    if (s != MR_OK) return s;
    if (K % MR_GEMV_K_MULTIPLE != 0 || M > mr::kShMaxM) return MR_ERR_UNSUPPORTED;
    const int cs = mr::route_cluster_size();
    mr::RoutePlan rp{};
    rp.cs = cs;
    rp.kc = K / cs;
    rp.clusters = 0;
    rp.ng = 1;
    rp.nl = 0;
    mr::RouteArgs a{};
    a.x = static_cast<const uint16_t*>(x);
    a.ldx = ldx;
    a.M = M;
    a.K = K;
    a.cs = cs;
    a.cs_shift = mr::ilog2_exact(cs);
    a.kc = K / cs;
    a.clusters = 0;
    a.flags = mr::launch_flags();
    a.wait_ns = mr::wait_limit_ns();
    if ((s = shared_args(w13, w13_scale, I, act, M, K, cs, &a, &rp)) != MR_OK) return s;
    mr::SharedPlan sp;
    mr::shared_plan(M, K, I, cs, &sp, mr::route_max_clusters());
    a.tok = sp.tok;
    a.tok_shift = mr::ilog2_exact(sp.tok);
    a.xpitch = sp.xpitch;
    return cuda_status(mr::launch_route_cluster(rp, a, as_stream(stream)));
}

}  // extern "C"
