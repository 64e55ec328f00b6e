// Plan and arguments of the cluster route kernel (route_kernel.cuh).
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace mr {

constexpr int kRouteThreads = 512;        // 16 warps per CTA
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kRouteBatch = 2;            // (tile, k-part) units whose loads a warp keeps in flight
constexpr int kRouteSpwMax = 8;           // 32-wide k steps per unit, at most
constexpr int kRouteSmemMax = 200 * 1024;    // dynamic shared memory, at most
constexpr int kRouteMaxM = 64;
constexpr int kRouteRowsPerCluster = 16;  // token rows per cluster of the whole route (one m16 MMA tile)
constexpr int kRouteGemvMaxM = 512;        // the router GEMV alone (above kRouteMaxM: tcgen05)
// Expert groups: routes over many experts split them across clusters (each
// cluster a group of >= kRouteGroupMinN experts) so that more SMs share the
// gate weight; the groups' top-k candidates meet in scratch.
constexpr int kRouteSplitMinN = 512;
constexpr int kRouteGroupMinN = 128;
constexpr int kRouteMaxGroups = 8;
// The router GEMV alone (no gate to merge) splits any N >= 32 into groups of
// >= 16 experts (two 8-expert MMA tiles), so that a 1.6 MB gate weight
// streams through up to 8 clusters instead of one.
constexpr int kRouteGemvGroupMinN = 16;

struct RouteArgs {
    const uint16_t* x;
    int64_t ldx;
    const uint16_t* w;
    const float* bias;
    float* logits;
    int32_t* ids;
    float* weights;
    int32_t* sorted;
    int32_t* expert_ids;
    int32_t* ntpp;
    int64_t capacity;
    uint8_t* q;
    uint8_t* scale;
    int M, N, K, topk, block, scoring, renormalize;
    int mode;        // 0: logits only, 1: whole route
    int cs;          // CTAs in the cluster
    int cs_shift;    // log2(cs)
    int rpc;         // token rows per cluster
    int clusters;    // clusters in the grid: one per 16 token rows
    int kc;          // K per CTA
    int spw;         // 32-wide k steps per unit
    int wpt;         // k-parts per 8-expert tile
    int units;       // (tile, part) units per CTA
    int tok;         // token rows owned per CTA
    int xpitch;      // bytes per x row in shared memory
    int off_x, off_recv, off_row, off_key, off_cand, off_ids, off_mask, off_start;
    int off_kred;    // wpt > 1: the k-parts' partial tiles handed to part 0 (two buffers)
    int tok_shift, wpt_shift;  // log2 of tok and wpt (both powers of two)
    int gs_shift;    // gate threshold: log2 of the lane-group size (<= 32 threads)
    int nslots;      // split-K partials per logit at the owner
    // q = (x * magic) >> 32 equals x / d for 0 <= x < 2^21, d <= 1024
    unsigned long long mag_n, mag_k, mag_block, mag_vpr, mag_n4;
    unsigned long long* trace;
    int flags;                   // launch flags (bit 1: test stall, see moe_route.h)
    unsigned long long wait_ns;  // limit of every wait for bytes from other CTAs
    int32_t* ids_scratch;   // clusters > 1: every token's ids, gathered for the sort
    unsigned* counter;      // clusters > 1: last-arriver ticket, zero between launches
    // expert groups (ng > 1): cluster cl takes token rows (cl / ng) * rpc ..
    // and experts (cl % ng) * N .. + N of ldn; N above is the group's width
    int ng, ldn;
    unsigned long long* cand_key;      // [M][ng][topk] selection composites, per group in rank order
    float* cand_val;                   // [M][ng][topk] their logits
    int off_merge;                     // shared memory of the merge (the CTA that arrives last)
    // router input on the norm's scale (rstd == nullptr: x is the router input
    // as given): x[m, k] -> bf16((x * rstd[m]) * s[k]), s = g or 1 + g
    const float* rstd;
    const uint16_t* norm_w;
    int norm_gemma;
    int quant_fp4;  // q holds MXFP4 ([M, K/2]) instead of MXFP8 ([M, K])
    // shared expert's gate/up projection + SwiGLU in the same launch
    // (sh_clusters > 0): the clusters after the route's each take sh_pairs
    // (gate row, up row) pairs of w13 (E4M3 [2 sh_I, K], rows [0, sh_I) gate)
    // with E8M0 scales [2 sh_I, K/32]; act = silu(gate) * up -> bf16 [M, sh_I]
    const uint8_t* sh_w;
    const uint8_t* sh_scale;
    uint16_t* sh_out;
    int sh_I, sh_clusters, sh_pairs, sh_wpt, sh_spw, sh_units, sh_nslots, sh_off_x, sh_off_recv;
    int sh_off_w, sh_off_s, sh_spitch;  // the CTA's weight slice and scale bytes in shared memory
};

// Multiplier for division by d (1 <= d <= 2^11) of dividends below 2^21:
// floor(x * ceil(2^32 / d) / 2^32) == floor(x / d).
inline unsigned long long div_magic(int d) {
    return (((unsigned long long)1 << 32) + (unsigned long long)d - 1) / (unsigned long long)d;
}
inline int ilog2_exact(int v) {
    int s = 0;
    while ((1 << s) < v) ++s;
    return (1 << s) == v ? s : -1;
}

struct RoutePlan {
    int cs, kc, spw, wpt, units, tok, xpitch, clusters, rpc;
    int sh_clusters;  // shared-expert clusters after the route's (0: none)
    int ng, nl, off_merge;  // expert groups, experts per group, merge buffers
    int nslots;
    bool half;
    int smem;
    int off_x, off_recv, off_row, off_key, off_cand, off_ids, off_mask, off_start, off_kred;
};

inline int align_up(int v, int a) { return (v + a - 1) / a * a; }

// Returns false when (M, N, K, topk) is outside what the cluster kernel
// covers with cluster size cs (at most kRouteMaxM rows, in both modes).
// max_groups: co-resident clusters available for expert groups (1: none).
inline bool route_plan(int M, int N, int K, int topk, int mode, int cs, RoutePlan* p, int max_groups = 1) {
    if (M < 1 || M > kRouteMaxM || N < 8 || N > 1024 || N % 8 != 0) return false;
    if (K < 32 * cs || K % (32 * cs) != 0) return false;
    RoutePlan q{};
    q.cs = cs;
    q.kc = K / cs;
    const int Ntot = N;
    q.ng = 1;
    // (the whole route splits one token group only: with several, the one
    // merging CTA takes several tokens per warp and the split measured slower)
    const int mcl = (M + kRouteRowsPerCluster - 1) / kRouteRowsPerCluster;
    const int split_min = mode == 0 ? 2 * kRouteGemvGroupMinN : kRouteSplitMinN;
    const int group_min = mode == 0 ? kRouteGemvGroupMinN : kRouteGroupMinN;
    if (max_groups > 1 && !(mode == 1 && mcl > 1) && N >= split_min) {
        int d = max_groups / mcl;
        if (d > kRouteMaxGroups) d = kRouteMaxGroups;
        for (; d >= 2; --d)
            if ((N / 8) % d == 0 && N / d >= group_min && topk <= N / d) break;
        if (d >= 2) q.ng = d;
    }
    N = Ntot / q.ng;  // from here on: the experts of one cluster
    q.nl = N;
    const int S = q.kc / 32, NT = N / 8;
    // k-parts per tile: a power of two (a warp keeps one part for all its
    // tiles) dividing S with at most kRouteSpwMax steps per part; more parts
    // while the CTA would have fewer tiles than warps WITHOUT expert groups
    // (the same split with and without groups: every logit then sums the
    // same partials in the same order, so the GEMV alone and the whole route
    // give the same bits however the experts are grouped)
    int w = 0;
    for (int d = 1; d <= kRouteWarps && d <= S; d *= 2)
        if (S % d == 0 && S / d <= kRouteSpwMax) {
            w = d;
            break;
        }
    if (w == 0) return false;
    const int NTall = Ntot / 8;
    while (NTall * w < kRouteWarps && 2 * w <= kRouteWarps && S % (2 * w) == 0) w *= 2;
    if (cs % 8 != 0) return false;  // the owner sums split-K slots in groups of 8
    q.wpt = w;
    q.spw = S / w;
    q.units = NT * w;
    // one cluster per 16 token rows; rows owned per CTA: a power of two
    // covering ceil(rows of a cluster / cs)
    q.rpc = kRouteRowsPerCluster;
    q.clusters = (M + q.rpc - 1) / q.rpc * q.ng;
    const int Mc = M < q.rpc ? M : q.rpc;
    q.tok = 1;
    while (q.tok * cs < Mc) q.tok *= 2;
    if (mode == 1 && (topk < 1 || topk > 32 || topk > N || q.tok > kRouteWarps)) return false;
    if (ilog2_exact(q.tok) < 0 || ilog2_exact(w) < 0 || ilog2_exact(cs) < 0) return false;
    q.half = M <= 8;
    q.xpitch = q.kc * 2 + (((q.kc * 2) % 128 == 0) ? 64 : 0);
    // (tcgen05 at 16 rows: a chain of K/16 dependent MMAs issued by one
    // thread plus the accumulator read-back measured slower than 16 warps of
    // mma.sync, so the decode route keeps mma.sync)
    // the CTA adds its k-parts before sending: one partial per CTA and logit
    q.nslots = cs;

    int off = 0;
    q.off_x = off;  // row-major x slice (MMA operand of mma.sync; quantiser input)
    off = align_up(off + Mc * q.xpitch, 16);
    q.off_recv = off;
    off = align_up(off + q.nslots * q.tok * N * 4, 16);
    q.off_row = off;
    off = align_up(off + q.tok * N * 4, 16);
    q.off_key = off;  // (unused: the selection keys stay in registers)
    q.off_cand = off;  // N candidate composites (one row at a time); per row k values; N exact scores
    off = align_up(off + (mode == 1 ? N * 12 + q.tok * topk * 8 : 0), 16);
    q.off_ids = off;  // every token's ids in the CTA that sorts
    off = align_up(off + M * (mode == 1 ? topk : 0) * 4, 16);
    q.off_mask = off;
    off = align_up(off + (mode == 1 ? Ntot : 0) * 8, 16);
    q.off_start = off;
    off = align_up(off + (mode == 1 ? Ntot + 32 : 0) * 4, 16);
    q.off_merge = off;  // ng > 1: the cluster's candidates as received (keys, then logits); in the
                        // merging CTA all candidates [M][ng][k] (8 B keys, then logits)
    if (mode == 1 && q.ng > 1) off = align_up(off + M * q.ng * topk * 12, 16);
    q.off_kred = off;  // [batch parity][warp][value][lane] floats, values: 4 (half) or 8 per lane
    if (w > 1) off = align_up(off + 2 * kRouteWarps * (q.half ? 4 : 8) * 32 * 4, 16);
    q.smem = off;
    if (q.smem > kRouteSmemMax) return false;
    *p = q;
    return true;
}

// Router GEMV alone for kRouteMaxM < M <= kRouteGemvMaxM rows on tcgen05:
// one cluster of cs CTAs per rpc token rows, CTA c the K slice c.  The
// slice arrives in stages of kTcStageK k (one 128-byte swizzled row per
// token or expert), all resident at once: per stage an rpc-row x tile (the
// MMA's N side) and a 128-row weight tile (its M side; rows past N are never
// written).  Offsets are from a 1024-byte aligned base inside the dynamic
// shared memory (1024 bytes of slack).  The split-K partials go through
// scratch: part_bytes of fp32 [clusters][cs][rpc][N].
constexpr int kTcStageK = 64;
constexpr int kTcWStageBytes = 128 * 128;
constexpr int kTcMaxStages = 8;
constexpr int kTcSmemMax = 226 * 1024;  // dynamic (the per-block maximum is 227 KiB with the static part)

struct TcGemvPlan {
    int cs, kc, nq, nstage, rpc, tok, clusters, tmem_cols, off_w, smem, part_bytes;
};

// Scratch bytes of the partials for any plan of M rows (any count of
// resident clusters): clusters * rpc < M + rpc <= M + 128 rows, cs <= 16.
inline int64_t tc_gemv_part_bound(int M, int N) { return (int64_t)(M + 127) * N * 16 * 4; }

// fit: clusters resident at once.  Rows per cluster: M spread over fit
// clusters, rounded up to a multiple of 16 (the MMA's N), 16 to 128: the
// fewer rows a cluster takes, the fewer bytes of x each CTA loads and of
// partials it sends (rpc x N fp32); the MMAs per CTA stay K / (16 cs).
// Returns false outside what the kernel covers.
inline bool tc_gemv_plan(int M, int N, int K, int cs, int fit, TcGemvPlan* p) {
    if (M <= kRouteMaxM || M > kRouteGemvMaxM || N < 8 || N > 128 || N % 8 != 0) return false;
    if (cs < 1 || K < cs || K % cs != 0 || (K / cs) % 16 != 0) return false;
    TcGemvPlan q{};
    q.cs = cs;
    q.kc = K / cs;
    q.nq = q.kc / 16;
    q.nstage = (q.kc + kTcStageK - 1) / kTcStageK;
    if (q.nstage > kTcMaxStages) return false;
    const int f = fit < 1 ? 1 : fit;
    q.rpc = ((M + f - 1) / f + 15) / 16 * 16;
    if (q.rpc < 16) q.rpc = 16;
    if (q.rpc > 128) q.rpc = 128;
    q.clusters = (M + q.rpc - 1) / q.rpc;
    q.tok = (q.rpc + cs - 1) / cs;  // rows whose logits each CTA sums (every CTA takes a share)
    q.tmem_cols = 32;  // fp32 accumulator: 128 lanes (experts) x rpc columns (tokens)
    while (q.tmem_cols < q.rpc) q.tmem_cols *= 2;
    const int xbytes = q.nstage * q.rpc * 128, wbytes = q.nstage * kTcWStageBytes;
    q.off_w = xbytes;
    q.smem = 1024 + xbytes + wbytes;
    q.part_bytes = q.clusters * q.rpc * N * cs * 4;
    if (q.smem > kTcSmemMax) return false;
    *p = q;
    return true;
}

// Shared expert's gate/up projection in the route launch (M <= 16 token rows,
// one cluster of cs CTAs per group of pairs, CTA c the K slice c as the
// route's): at most kShUnitsPerWarp (8-row tile, k-part) units per warp.
constexpr int kShUnitsPerWarp = 4;
constexpr int kShMaxClusters = 16;  // (clusters never wait on each other: more than fit at once is fine)
constexpr int kShMaxM = 16;
constexpr int kShScaleBatch = 8;  // scale-byte loads a thread keeps in flight

struct SharedPlan {
    int clusters, pairs, wpt, spw, units, nslots, tok, xpitch, off_x, off_recv, off_w, off_s, spitch, smem;
};

// Returns false when (M, K, I) is outside what the shared-expert CTAs cover.
// fit: clusters that can run beside the route's at once; the plan takes the
// most clusters up to fit (one wave), else the fewest beyond it.
inline bool shared_plan(int M, int K, int I, int cs, SharedPlan* p, int fit = kShMaxClusters) {
    if (M < 1 || M > kShMaxM || I < 8 || I % 8 != 0 || K < 32 * cs || K % (32 * cs) != 0) return false;
    SharedPlan q{};
    const int kc = K / cs, S = kc / 32;
    int w = 0;
    for (int d = 1; d <= kRouteWarps && d <= S; d *= 2)
        if (S % d == 0 && S / d <= kRouteSpwMax) {
            w = d;
            break;
        }
    if (w == 0 || (cs * w) % 8 != 0) return false;
    // clusters: a divisor of the 8-pair groups with at most kShUnitsPerWarp
    // units per warp; the most that fit at once, else the fewest that work
    auto ok = [&](int d) {
        return (I / 8) % d == 0 && (2 * (I / d) / 8) * w <= kShUnitsPerWarp * kRouteWarps &&
               2 * (I / d) <= kRouteThreads;  // a thread per row loads the scales
    };
    int sc = 0;
    for (int d = fit < kShMaxClusters ? fit : kShMaxClusters; d >= 1 && sc == 0; --d)
        if (ok(d)) sc = d;
    for (int d = (fit < kShMaxClusters ? fit : kShMaxClusters) + 1; d <= kShMaxClusters && sc == 0; ++d)
        if (ok(d)) sc = d;
    if (sc == 0) return false;
    q.clusters = sc;
    q.pairs = I / sc;
    q.wpt = w;
    q.spw = S / w;
    q.units = (2 * q.pairs / 8) * w;
    q.nslots = cs * w;
    q.tok = 1;
    while (q.tok * cs < M) q.tok *= 2;
    q.xpitch = kc * 2 + (((kc * 2) % 128 == 0) ? 64 : 0);
    int off = 0;
    q.off_x = off;
    off = align_up(off + M * q.xpitch, 16);
    q.off_recv = off;
    off = align_up(off + q.nslots * q.tok * 2 * q.pairs * 4, 16);
    q.off_w = off;  // 2P rows of kc weight bytes, 16 bytes of padding a row
    off = align_up(off + 2 * q.pairs * (kc + 16), 16);
    q.spitch = align_up(kc / 32, 4);
    q.off_s = off;  // 2P rows of kc / 32 scale bytes
    off = align_up(off + 2 * q.pairs * q.spitch, 16);
    q.smem = off;
    if (q.smem > kRouteSmemMax) return false;
    *p = q;
    return true;
}

}  // namespace mr
