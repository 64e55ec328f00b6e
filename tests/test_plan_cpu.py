"""Host logic of the route kernel's plan (csrc/route_plan.h), compiled here
with the host C++ compiler: for a grid of shapes every plan the kernel can
receive keeps the invariants its index arithmetic relies on."""

import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROBE = r'''
#include <cstdio>
#include <initializer_list>
#include "route_plan.h"
int main() {
    const int Ms[] = {1, 2, 3, 4, 7, 8, 9, 15, 16, 17, 31, 32, 33, 47, 63, 64, 65, 100};
    const int Ns[] = {8, 40, 64, 128, 136, 256, 512, 640, 896, 1024};
    const int Ks[] = {512, 1024, 3584, 6144, 7168};
    const int topks[] = {1, 4, 8, 16, 32};
    for (int mg : {1, 7, 9})
    for (int mode = 0; mode < 2; ++mode)
    for (int M : Ms) for (int N : Ns) for (int K : Ks) for (int k : topks) {
        if (k > N) continue;
        mr::RoutePlan p;
        if (!mr::route_plan(M, N, K, k, mode, 16, &p, mg)) { printf("none %d %d %d %d %d %d\n", mg, mode, M, N, K, k); continue; }
        printf("plan %d %d %d %d %d %d ng=%d nl=%d clusters=%d rpc=%d tok=%d wpt=%d spw=%d nslots=%d smem=%d cs=%d kc=%d half=%d\n",
               mg, mode, M, N, K, k, p.ng, p.nl, p.clusters, p.rpc, p.tok, p.wpt, p.spw, p.nslots, p.smem, p.cs,
               p.kc, (int)p.half);
    }
}
'''


@pytest.fixture(scope="module")
def plans(tmp_path_factory):
    d = tmp_path_factory.mktemp("plan")
    src = d / "probe.cpp"
    src.write_text(PROBE)
    exe = d / "probe"
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", os.path.join(ROOT, "decode_expert_routing_gb300", "csrc"),
                    "-o", str(exe), str(src)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines()
    res = []
    for line in out:
        parts = line.split()
        key = tuple(int(v) for v in parts[1:7])
        if parts[0] == "none":
            res.append((key, None))
        else:
            res.append((key, {kv.split("=")[0]: int(kv.split("=")[1]) for kv in parts[7:]}))
    return res


def test_plans_keep_the_kernel_invariants(plans):
    pow2 = lambda v: v > 0 and (v & (v - 1)) == 0
    n_plans = 0
    for (mg, mode, M, N, K, k), p in plans:
        if p is None:
            continue
        n_plans += 1
        assert p["cs"] == 16 and p["kc"] * 16 == K and p["kc"] % 32 == 0
        assert p["nl"] * p["ng"] == N and p["nl"] % 8 == 0
        if p["ng"] > 1:  # expert groups: >= 128 experts for the whole route, >= 16 for the GEMV alone
            assert mg > 1 and (N >= 512 and p["nl"] >= 128 and k <= p["nl"] if mode == 1 else p["nl"] >= 16)
        if mode == 1 and p["ng"] > 1:
            assert M <= 16                       # the whole route splits one token group only
        assert p["clusters"] == -(-M // p["rpc"]) * p["ng"]
        assert p["ng"] == 1 or p["clusters"] <= max(mg, 1)
        assert pow2(p["tok"]) and pow2(p["wpt"]) and p["tok"] * 16 >= min(M, p["rpc"])
        assert p["wpt"] * p["spw"] * 32 == p["kc"] and p["spw"] <= 8
        assert p["nslots"] % 8 == 0
        assert p["smem"] <= 200 * 1024 and p["smem"] % 16 == 0
        assert p["half"] == (1 if M <= 8 else 0)
        assert M <= 64 and p["rpc"] == 16          # above 64 rows: the tensor-core GEMV's own plan
        if mode == 1:
            assert p["tok"] <= 16
    assert n_plans > 1000


def test_every_documented_decode_shape_has_a_plan(plans):
    have = {key for key, p in plans if p is not None}
    for M in (1, 2, 4, 8, 16, 32, 64):
        assert (9, 1, M, 128, 6144, 8) in have
    for M in (1, 8, 16, 32):
        assert (9, 1, M, 896, 3584, 16) in have
    assert not any(key[2] > 64 for key in have)


def test_expert_groups_keep_the_split_k_of_the_unsplit_plan(plans):
    """Every logit sums the same split-K partials in the same order whether
    or not the experts are split into groups, and in the GEMV alone as in the
    whole route (M <= 64): the k-parts per tile, the k-steps per part and the
    slots per logit agree, so the logits are the same bits."""
    by_key = {key: p for key, p in plans if p is not None}
    n = 0
    for (mg, mode, M, N, K, k), p in by_key.items():
        ref = by_key.get((1, mode, M, N, K, k))
        if ref is not None:
            assert (p["wpt"], p["spw"], p["nslots"]) == (ref["wpt"], ref["spw"], ref["nslots"])
            n += p["ng"] > 1
        route = by_key.get((mg, 1, M, N, K, k))
        if mode == 0 and route is not None:
            assert (p["wpt"], p["spw"], p["nslots"]) == (route["wpt"], route["spw"], route["nslots"])
    assert n > 100


SHARED_PROBE = r"""
#include <cstdio>
#include <initializer_list>
#include "route_plan.h"
int main() {
    for (int cs : {8, 16})
    for (int M = 1; M <= 17; ++M)
    for (int K : {512, 3584, 6144, 7168})
    for (int I : {8, 64, 96, 256, 768, 1024, 1536, 2048, 100}) {
        mr::SharedPlan p;
        if (!mr::shared_plan(M, K, I, cs, &p)) { printf("none %d %d %d %d\n", cs, M, K, I); continue; }
        printf("plan %d %d %d %d %d %d %d %d %d %d %d %d\n", cs, M, K, I, p.clusters, p.pairs, p.wpt, p.spw,
               p.units, p.nslots, p.tok, p.smem);
        mr::SharedPlan q;  // one wave beside a route cluster on a device with 7 co-resident clusters
        if (cs == 16 && K == 6144 && I == 768 && mr::shared_plan(M, K, I, cs, &q, 6) && q.clusters != 6)
            printf("bad %d\n", q.clusters);
    }
}
"""


def test_shared_plan_invariants(tmp_path):
    """Every shared-expert plan keeps what the kernel's indexing relies on:
    pairs in whole 8-row tiles split evenly over the clusters, at most four
    units per warp, the K slice covered by the parts, the owners' token rows,
    split-K slots in groups of 8, shared memory within the route kernel's."""
    src = tmp_path / "probe.cpp"
    src.write_text(SHARED_PROBE)
    exe = tmp_path / "probe"
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", os.path.join(ROOT, "decode_expert_routing_gb300", "csrc"),
                    "-o", str(exe), str(src)], check=True)
    lines = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines()
    n = 0
    for line in lines:
        f = line.split()
        cs, M, K, I = (int(v) for v in f[1:5])
        S = K // cs // 32 if K % (32 * cs) == 0 else 0
        w = next((d for d in (1, 2, 4, 8, 16) if S and S % d == 0 and S // d <= 8), 0)
        fits = [d for d in range(1, 17) if I % 8 == 0 and (I // 8) % d == 0 and (2 * (I // d) // 8) * w <= 64
                and 2 * (I // d) <= 512]
        if f[0] == "none":
            assert M > 16 or I % 8 or not S or not w or not fits
            continue
        sc, P, w2, spw, units, nslots, tok, smem = (int(v) for v in f[5:])
        n += 1
        assert w2 == w and sc == max(fits)
        assert sc * P == I and P % 8 == 0 and 1 <= sc <= 16
        assert units == (2 * P // 8) * w and units <= 4 * 16
        assert w * spw * 32 * cs == K and spw <= 8 and nslots == cs * w and nslots % 8 == 0
        assert tok * cs >= M and tok & (tok - 1) == 0
        assert smem <= 200 * 1024 and smem >= 2 * P * (K // cs + 16)  # the staged weight slice fits
    assert n > 300
    assert not any(line.startswith("bad") for line in lines)
    have = {tuple(int(v) for v in line.split()[1:5]) for line in lines if line.startswith("plan")}
    for M in range(1, 17):
        assert (16, M, 6144, 768) in have and (16, M, 6144, 1536) in have and (8, M, 6144, 768) in have


TC_PROBE = r"""
#include <cstdio>
#include <initializer_list>
#include "route_plan.h"
int main() {
    for (int cs : {8, 16})
    for (int fit : {1, 4, 7, 8, 16})
    for (int M : {1, 64, 65, 100, 128, 129, 200, 256, 300, 448, 449, 512, 513})
    for (int N : {8, 40, 64, 120, 128, 136, 1024})
    for (int K : {512, 1024, 3584, 6144, 7168, 8192}) {
        mr::TcGemvPlan p;
        if (!mr::tc_gemv_plan(M, N, K, cs, fit, &p)) { printf("none %d %d %d %d %d\n", cs, fit, M, N, K); continue; }
        printf("plan %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %lld\n", cs, fit, M, N, K, p.kc, p.nq, p.nstage,
               p.rpc, p.tok, p.clusters, p.tmem_cols, p.off_w, p.smem, p.part_bytes,
               (long long)mr::tc_gemv_part_bound(M, N));
    }
}
"""


def test_tc_gemv_plan_invariants(tmp_path):
    """Every plan of the tensor-core GEMV (64 < M <= 512, N <= 128) keeps
    what the kernel relies on: whole 16-wide k-steps per CTA, at most 8
    resident 64-wide stages, 1024-byte aligned swizzled stage tiles, rows per
    cluster a multiple of 16 spreading M over the resident clusters (one
    wave), the owners' token rows, the accumulator's columns, and partials
    within the scratch bound the library sizes scratch by."""
    src = tmp_path / "probe.cpp"
    src.write_text(TC_PROBE)
    exe = tmp_path / "probe"
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", os.path.join(ROOT, "decode_expert_routing_gb300", "csrc"),
                    "-o", str(exe), str(src)], check=True)
    lines = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines()
    pow2 = lambda v: v > 0 and (v & (v - 1)) == 0
    have = {}
    for line in lines:
        f = line.split()
        cs, fit, M, N, K = (int(v) for v in f[1:6])
        if f[0] == "none":
            kc = K // cs
            rpc = min(128, max(16, -(-(-(-M // fit)) // 16) * 16))
            assert (M <= 64 or M > 512 or N > 128 or N % 8 or K % cs or kc % 16
                    or -(-kc // 64) > 8 or 1024 + (rpc * 128 + 16384) * -(-kc // 64) > 226 * 1024)
            continue
        kc, nq, nstage, rpc, tok, clusters, tcols, off_w, smem, part, bound = (int(v) for v in f[6:])
        have[(cs, fit, M, N, K)] = dict(rpc=rpc, clusters=clusters, smem=smem)
        assert 64 < M <= 512 and N <= 128 and N % 8 == 0
        assert kc * cs == K and kc % 16 == 0 and nq == kc // 16 and nstage == -(-kc // 64) <= 8
        assert rpc == min(128, max(16, -(-(-(-M // fit)) // 16) * 16)) and clusters == -(-M // rpc)
        assert clusters <= fit or rpc == 128                       # one wave whenever 128-row clusters allow it
        assert tok == -(-rpc // cs)                                # every CTA sums a share of the rows
        assert pow2(tcols) and tcols >= max(32, rpc) and tcols < 2 * max(32, rpc)
        assert off_w == nstage * rpc * 128 and off_w % 1024 == 0 and (rpc * 128) % 1024 == 0
        assert smem == 1024 + off_w + nstage * 16384 and smem <= 226 * 1024
        assert part == clusters * rpc * N * cs * 4 and part <= bound
    big = have[(16, 7, 512, 128, 6144)]
    assert big["rpc"] == 80 and big["clusters"] == 7           # one wave where 64-row clusters would need 8
    assert have[(16, 7, 448, 128, 6144)]["rpc"] == 64 and have[(16, 7, 128, 128, 6144)]["clusters"] == 4
    for M in (65, 128, 256, 512):
        assert (16, 7, M, 128, 6144) in have and (16, 7, M, 128, 7168) in have
