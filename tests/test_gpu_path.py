"""GPU parity of every step of the routing path against the CPU oracle.

Logits: |gpu - ref| <= 1e-4 * (1 + |ref|) against the oracle's fp64 dot
products.  Ids, sort outputs, e4m3 codes and e8m0 scales: bit-exact, with the
gate and the sort checked on the GPU's own logits and ids (so fp32 summation
order cannot flip a near-tie).  Weights: within 1e-6.
"""

import numpy as np
import pytest

import oracle
from decode_expert_routing_gb300 import inputs
from tests.gpu_util import (assert_logits_close, check_gate, check_quant, check_sort, host,
                            to_dev, to_dev_bf16, torch_mod)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mr():
    from decode_expert_routing_gb300 import build
    build.build()
    import decode_expert_routing_gb300 as m
    m.load_library()
    return m


def _cfg_cases():
    cases = []
    for cid in (1, 2, 3, 4, 5):
        c = inputs.CONFIGS[cid]
        for M in c["Ms"]:
            cases.append((cid, M))
    return cases


# ------------------------------------------------------------------ GEMV


@pytest.mark.parametrize("cid,M", _cfg_cases())
def test_router_gemv_matches_oracle(mr, cid, M):
    c = inputs.CONFIGS[cid]
    x, w = inputs.router_inputs(M, c["K"], c["N"], cid)
    if cid == 4:
        x = inputs.prefill_x(M, c["K"])
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    scratch = mr.Scratch(M, c["N"], c["K"], c["topk"])
    g1 = mr.router_gemv(xd, wd, scratch=scratch)
    g2 = mr.router_gemv(xd, wd, scratch=scratch)
    ref = oracle.router_gemv(x, w)
    assert_logits_close(host(g1), ref)
    assert np.array_equal(host(g1).view(np.uint32), host(g2).view(np.uint32)), "not deterministic"
    assert int(scratch.counters().abs().sum()) == 0, "split-K counters not re-zeroed"


@pytest.mark.parametrize("M,legacy", [(65, 0), (100, 0), (129, 0), (200, 0), (512, 0), (100, 1), (512, 1)])
def test_router_gemv_rows_past_64(mr, M, legacy):
    """More than 64 rows: the tensor-core GEMV (ragged last cluster), or with
    the legacy launch option the split-K mma.sync GEMV with last-arriver
    fixup."""
    x, w = inputs.router_inputs(M, 6144, 128, 7)
    scratch = mr.Scratch(M, 128, 6144, 8)
    flags = mr.get_launch_flags()
    if legacy:
        mr.set_launch_flags(flags | mr.LAUNCH_LEGACY_MMA)
    try:
        g = mr.router_gemv(to_dev_bf16(x), to_dev_bf16(w), scratch=scratch)
    finally:
        mr.set_launch_flags(flags)
    assert_logits_close(host(g), oracle.router_gemv(x, w))
    assert int(scratch.counters().abs().sum()) == 0


@pytest.mark.parametrize("M", [100, 300])
def test_router_gemv_split_k_ticket_path(mr, M):
    """Shapes the cluster kernel cannot hold in shared memory (N = 1024)
    take the split-K GEMV with last-arriver fixup; its counters re-zero."""
    x, w = inputs.router_inputs(M, 6144, 1024, 7)
    scratch = mr.Scratch(M, 1024, 6144, 8)
    g = mr.router_gemv(to_dev_bf16(x), to_dev_bf16(w), scratch=scratch)
    assert_logits_close(host(g), oracle.router_gemv(x, w))
    assert int(scratch.counters().abs().sum()) == 0


def test_router_gemv_strided_x(mr):
    M, K, N = 5, 6144, 128
    x, w = inputs.router_inputs(M, K, N, 21)
    xp = np.zeros((M, K + 64), np.uint16)
    xp[:, :K] = x
    xd = to_dev_bf16(xp)[:, :K]
    assert xd.stride(0) == K + 64
    g = mr.router_gemv(xd, to_dev_bf16(w))
    assert_logits_close(host(g), oracle.router_gemv(x, w))


def test_router_gemv_tied_rows_bitwise(mr):
    """Identical gate rows give bitwise-identical logits (same k partition
    and order for every expert)."""
    x, w = inputs.router_inputs(64, 6144, 128, 5)
    w = inputs.tied_gate(w)
    for M in (1, 8, 16, 64):
        g = host(mr.router_gemv(to_dev_bf16(x[:M]), to_dev_bf16(w))).view(np.uint32)
        assert np.array_equal(g[:, 10], g[:, 11]) and np.array_equal(g[:, 50], g[:, 51])


# ------------------------------------------------------------------ gate


@pytest.mark.parametrize("cid,M", [(1, 1), (2, 2), (2, 16), (2, 64), (3, 1), (3, 8), (3, 16),
                                   (3, 32), (4, 512)])
def test_gate_matches_oracle_on_gpu_logits(mr, cid, M):
    c = inputs.CONFIGS[cid]
    x, w = inputs.router_inputs(M, c["K"], c["N"], cid)
    bias = inputs.selection_bias(c["N"]) if c["scoring"] == "sigmoid" else None
    logits = mr.router_gemv(to_dev_bf16(x), to_dev_bf16(w))
    ids, wts = mr.route_topk(logits, c["topk"], c["scoring"], None if bias is None else to_dev(bias))
    lh = host(logits)
    check_gate(lh, host(ids), host(wts), c["topk"], c["scoring"], bias)
    # informational: how often the oracle's own logits would pick other ids
    rid, _ = oracle.route_topk(oracle.router_gemv(x, w), c["topk"], c["scoring"], bias)
    flips = int(np.sum(np.any(np.sort(rid, 1) != np.sort(host(ids), 1), 1)))
    print(f"config {cid} M={M}: rows whose selection differs on oracle logits: {flips}/{M}")


@pytest.mark.parametrize("scoring", ["softmax", "sigmoid"])
@pytest.mark.parametrize("renorm", [True, False])
def test_gate_modes_and_edges(mr, scoring, renorm):
    rng = np.random.default_rng(3)
    for N, k in ((8, 1), (8, 8), (128, 8), (256, 32), (896, 16), (1024, 32), (40, 7)):
        lg = (rng.standard_normal((9, N)) * 2).astype(np.float32)
        lg[0] = 0.25                                  # all equal
        lg[1, ::2] = -0.0                             # signed zeros tie with +0
        lg[1, 1::2] = 0.0
        lg[2, : N // 2] = lg[2, N // 2: 2 * (N // 2)]  # pairwise ties
        bias = (rng.uniform(-0.1, 0.1, N)).astype(np.float32)
        ids, wts = mr.route_topk(to_dev(lg), k, scoring, to_dev(bias) if scoring == "sigmoid" else None,
                                 renormalize=renorm)
        check_gate(lg, host(ids), host(wts), k, scoring, bias if scoring == "sigmoid" else None, renorm)


def _hard_sigmoid_logits():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "sigmoid_hard_cases.txt")
    rows = [ln.split() for ln in open(path) if not ln.startswith("#")]
    return np.array([int(r[0], 16) for r in rows], dtype=np.uint32).view(np.float32)


def _sigmoid_scores_on_gpu(mr, lg):
    """The kernel's sigmoid score of every logit: with k = N = 32 every expert
    is selected, and the weights without renormalisation are the scores."""
    ids, wts = mr.route_topk(to_dev(lg), 32, "sigmoid", None, renormalize=False)
    ids, wts = host(ids), host(wts)
    return wts, np.take_along_axis(lg, ids, 1)


def _sigmoid_sweep(n_rows):
    rng = np.random.default_rng(17)
    vals = np.concatenate([np.linspace(-88, 88, n_rows * 32 - 4096), rng.uniform(-110, -87, 2048),
                           rng.uniform(15, 40, 2048)]).astype(np.float32)
    rng.shuffle(vals)
    hard = _hard_sigmoid_logits()
    vals[: hard.size] = hard
    return vals.reshape(n_rows, 32)


@pytest.mark.parametrize("slow", [False, True])
def test_sigmoid_scores_correctly_rounded_bitwise(mr, slow):
    """The kernel's sigmoid scores equal the oracle's correctly rounded fp32
    sigmoid bit for bit: over 2^20 logits in [-88, 88] plus the subnormal and
    near-one ranges and the stored hard cases (within ~1e-14 of an fp32
    rounding boundary, where the fp64 path's rounding test fails and the
    double-double path decides).  slow: the test hook that sends every score
    through the double-double path (a smaller sweep)."""
    lg = _sigmoid_sweep(1 << 10 if slow else 1 << 15)
    prev = mr.get_launch_flags()
    mr.set_launch_flags(prev | (mr.LAUNCH_TEST_SLOW_SIGMOID if slow else 0))
    try:
        wts, picked = _sigmoid_scores_on_gpu(mr, lg)
    finally:
        mr.set_launch_flags(prev)
    want = oracle.sigmoid_f32(picked)
    bad = np.flatnonzero(wts.view(np.uint32).ravel() != want.view(np.uint32).ravel())
    assert bad.size == 0, [(float(picked.ravel()[i]), float(wts.ravel()[i]), float(want.ravel()[i])) for i in bad[:5]]


def _near_tie_bias(lg_rows, bias, k, offset_ulps):
    """Bias of the expert ranked k+1 on row 0 moved so that its exact key
    (oracle sigmoid + bias, fp32) sits offset_ulps from the k-th key: 0 is an
    exact tie (the lower id wins), +-1 one ulp above or below.  The
    approximate fp32 scores cannot order such keys; only exact ones can."""
    s = oracle.sigmoid_f32(lg_rows[0])
    t = (s + bias).astype(np.float32)
    order = np.lexsort((np.arange(t.size), -t.astype(np.float64)))
    i, j = int(order[k - 1]), int(order[k])
    target = t[i]
    for _ in range(abs(offset_ulps)):
        target = np.nextafter(target, np.float32(np.inf if offset_ulps > 0 else -np.inf))
    b = bias.copy()
    bj = np.float32(np.float64(target) - np.float64(s[j]))
    for _ in range(64):  # nearest bias with s_j + b_j == target in fp32
        got = np.float32(s[j] + bj)
        if got == target:
            break
        bj = np.nextafter(bj, np.float32(np.inf if got < target else -np.inf))
    assert np.float32(s[j] + bj) == target
    b[j] = bj
    return b


@pytest.mark.parametrize("offset", [-1, 0, 1])
def test_sigmoid_near_ties_decided_by_exact_scores(mr, offset):
    """Keys one ulp apart or tied (the k-th and (k+1)-th of a token, built by
    moving one bias): the standalone gate and the one-launch route pick the
    oracle's ids, bit for bit, on the GPU's logits."""
    K, N, k, B = 3584, 896, 16, 16
    for M in (1, 8):
        x, w = inputs.router_inputs(M, K, N, 3)
        xd, wd = to_dev_bf16(x), to_dev_bf16(w)
        lh = host(mr.router_gemv(xd, wd))
        bias = _near_tie_bias(lh, inputs.selection_bias(N), k, offset)
        ids, wts = mr.route_topk(to_dev(lh), k, "sigmoid", to_dev(bias))
        check_gate(lh, host(ids), host(wts), k, "sigmoid", bias)
        out = mr.moe_route_sort_quant(xd, wd, k, B, "sigmoid", to_dev(bias))
        assert np.array_equal(host(out["logits"]).view(np.uint32), lh.view(np.uint32))
        check_gate(lh, host(out["topk_ids"]), host(out["topk_weights"]), k, "sigmoid", bias)


def test_route_sigmoid_slow_path_same_bits(mr):
    """The one-launch route over 896 experts with every exact score taken by
    the double-double path gives the same bits as the normal path."""
    K, N, k, B = 3584, 896, 16, 16
    x, w = inputs.router_inputs(8, K, N, 3)
    bias = to_dev(inputs.selection_bias(N))
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    ref = mr.moe_route_sort_quant(xd, wd, k, B, "sigmoid", bias)
    prev = mr.get_launch_flags()
    mr.set_launch_flags(prev | mr.LAUNCH_TEST_SLOW_SIGMOID)
    try:
        got = mr.moe_route_sort_quant(xd, wd, k, B, "sigmoid", bias)
        torch_mod().cuda.synchronize()
    finally:
        mr.set_launch_flags(prev)
    for name in ("logits", "topk_ids", "topk_weights", "sorted_token_ids", "expert_ids", "q", "scale"):
        a, b = host(ref[name]), host(got[name])
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), name


# ------------------------------------------------------------------ sort


@pytest.mark.parametrize("M,k,N,B", [(1, 8, 128, 16), (2, 8, 128, 16), (16, 8, 128, 16), (64, 8, 128, 16),
                                     (32, 16, 896, 16), (16, 16, 896, 16), (256, 8, 128, 16), (4096, 8, 128, 64),
                                     (257, 8, 128, 64), (7, 3, 9, 1), (100, 32, 1024, 128), (333, 7, 50, 32),
                                     (8192, 8, 128, 64), (9000, 8, 128, 16), (2100, 32, 1024, 16)])
def test_sort_matches_oracle(mr, M, k, N, B):
    rng = np.random.default_rng(M * 7 + k)
    ids = np.stack([rng.permutation(N)[:k] for _ in range(M)]).astype(np.int32)
    st, ex, nt = mr.moe_sort(to_dev(ids), N, B)
    check_sort(ids, N, B, host(st), host(ex), host(nt))


def test_sort_masked_and_skewed_ids(mr):
    rng = np.random.default_rng(11)
    for M in (16, 64, 300, 4096):
        ids = rng.integers(0, 4, size=(M, 8)).astype(np.int32)     # heavy skew, repeats
        ids[::3, 0] = -1                                          # masked
        ids[::5, 1] = 130                                         # out of range (N=128)
        st, ex, nt = mr.moe_sort(to_dev(ids), 128, 16)
        check_sort(ids, 128, 16, host(st), host(ex), host(nt))


def test_sort_prefill_on_gate_ids(mr):
    """Config 4 prefill: the ids come from the gate of the GEMV of the same x."""
    c = inputs.CONFIGS[4]
    M = c["prefill_M"]
    x = inputs.prefill_x(M, c["K"])
    _, w = inputs.router_inputs(8, c["K"], c["N"], 4)
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    logits = mr.router_gemv(xd[:512], wd)          # GEMV covers <= 512 rows per call
    parts = [logits]
    for r in range(512, M, 512):
        parts.append(mr.router_gemv(xd[r:r + 512], wd))
    import torch
    logits = torch.cat(parts)
    ids, _ = mr.route_topk(logits, c["topk"])
    scratch = mr.Scratch(M, c["N"], c["K"], c["topk"])
    st, ex, nt = mr.moe_sort(ids, c["N"], c["block"], scratch=scratch)
    check_sort(host(ids), c["N"], c["block"], host(st), host(ex), host(nt))
    assert int(scratch.counters().abs().sum()) == 0


# ------------------------------------------------------------------ quant


@pytest.mark.parametrize("what", ["decode64", "prefill4096", "edges", "large_expert"])
def test_quant_matches_oracle(mr, what):
    if what == "decode64":
        x, _ = inputs.router_inputs(64, 6144, 8, 2)
    elif what == "prefill4096":
        x = inputs.prefill_x(4096, 6144)
    elif what == "edges":
        x = inputs.quant_edge_x(64, 6144)
    else:
        x, _ = inputs.router_inputs(32, 3584, 8, 3)
    q, s = mr.mxfp8_quant(to_dev_bf16(x))
    check_quant(x, host(q), host(s))


def test_quant_exhaustive_bf16_patterns(mr):
    """Every finite bf16 pattern, in blocks whose amax pins the scale to a
    chosen exponent, against the oracle."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    pats = pats[(pats & 0x7F80) != 0x7F80]
    rows = []
    for anchor in (0x0001, 0x0080, 0x3F80, 0x43E0, 0x43DF, 0x4400, 0x7F7F):
        a_mag = anchor & 0x7FFF
        vals = pats[(pats & 0x7FFF) <= a_mag]
        n = (len(vals) + 30) // 31 * 31
        vals = np.concatenate([vals, np.zeros(n - len(vals), np.uint16)]).reshape(-1, 31)
        blocks = np.concatenate([np.full((len(vals), 1), anchor, np.uint16), vals], 1)
        rows.append(blocks.reshape(-1))
    flat = np.concatenate(rows)
    K = 6144
    flat = np.concatenate([flat, np.zeros((-len(flat)) % K, np.uint16)]).reshape(-1, K)
    q, s = mr.mxfp8_quant(to_dev_bf16(flat))
    check_quant(flat, host(q), host(s))


def test_quant_past_int32_offsets(mr):
    """M*K beyond 2^31 elements (past the int32 offset limit the MiniMax-M3.1
    sort PR names for hidden 6144): rows past the limit quantise exactly like
    the rows they copy."""
    import torch
    K, limit = 6144, (2 ** 31) // 6144
    M = limit + 3
    base, _ = inputs.router_inputs(97, K, 8, 4)
    xd = to_dev_bf16(base).repeat((M + 96) // 97, 1)[:M].contiguous()
    q, s = mr.mxfp8_quant(xd)
    torch.cuda.synchronize()
    rq, rs = oracle.mxfp8_quant(base)
    for r in (0, 1, limit - 1, limit, limit + 1, M - 1):
        assert np.array_equal(host(q[r]), rq[r % 97]), r
        assert np.array_equal(host(s[r]), rs[r % 97]), r
    del xd, q, s
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ config 5


def test_adversarial_skew_ties_and_quant_edges(mr):
    import torch
    c = inputs.CONFIGS[5]
    M, K, N, k, B = 64, c["K"], c["N"], c["topk"], c["block"]
    x, w = inputs.router_inputs(M, K, N, 5)
    w = inputs.tied_gate(w)
    x = inputs.quant_edge_x(M, K)
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    logits = mr.router_gemv(xd, wd)
    assert_logits_close(host(logits), oracle.router_gemv(x, w))
    lg = host(logits).view(np.uint32)
    assert np.array_equal(lg[:, 10], lg[:, 11]) and np.array_equal(lg[:, 50], lg[:, 51])
    # (a) skew: +3 on experts 0..3, applied to the logits between GEMV and gate
    logits[:, :4] += 3.0
    ids, wts = mr.route_topk(logits, k)
    lh = host(logits)
    rid, _ = check_gate(lh, host(ids), host(wts), k, "softmax")
    # (b) ties: wherever 11 (or 51) is chosen, 10 (or 50) is chosen before it
    for row in rid:
        row = row.tolist()
        for a, b in ((10, 11), (50, 51)):
            if b in row:
                assert a in row and row.index(a) < row.index(b)
    st, ex, nt = mr.moe_sort(ids, N, B)
    check_sort(host(ids), N, B, host(st), host(ex), host(nt))
    hist = np.bincount(host(ids).reshape(-1), minlength=N)
    print(f"skew: experts 0-3 take {hist[:4].sum() / hist.sum():.1%} of assignments, "
          f"{int(np.sum(hist == 0))} experts empty")
    # (c) quantiser edge blocks
    q, s = mr.mxfp8_quant(xd)
    check_quant(x, host(q), host(s))
    torch.cuda.synchronize()


def test_scratch_dirty_check_refuses_before_launch(mr):
    """With the debug scratch check on, a call whose scratch counters are not
    zero (one slot corrupted from the host) returns MR_ERR_SCRATCH_DIRTY and
    launches nothing (its output keeps its sentinel); after a reset the same
    calls succeed.  Covers the split-K GEMV, the multi-CTA sort and the
    one-launch route over several clusters (the sort above 65536
    assignments, where it takes two launches)."""
    torch = torch_mod()
    N, K, k, B = 128, 6144, 8, 16
    prev = mr.get_launch_flags()
    x, w = inputs.router_inputs(128, K, N, 2)
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    scratch = mr.Scratch(512, N, K, k)
    ids = to_dev(np.random.default_rng(1).integers(0, N, (9000, k)).astype(np.int32))  # > 65536: two launches
    calls = {
        "gemv": lambda: mr.router_gemv(xd, wd, out=lg, scratch=scratch),
        "sort": lambda: mr.moe_sort(ids, N, B, scratch=scratch),
        "route": lambda: mr.moe_route_sort_quant(xd[:32], wd, k, B, scratch=scratch),
    }
    lg = torch.full((128, N), float("nan"), dtype=torch.float32, device="cuda")
    try:
        mr.set_launch_flags(prev | mr.LAUNCH_CHECK_SCRATCH | mr.LAUNCH_LEGACY_MMA)
        for name, fn in calls.items():
            scratch.counters()[4097 if name == "sort" else 17] = 5
            torch.cuda.synchronize()
            with pytest.raises(mr.MoeRouteError) as ei:
                fn()
            assert ei.value.status == mr.MR_ERR_SCRATCH_DIRTY, name
            scratch.reset()
            fn()
            torch.cuda.synchronize()
            assert int(scratch.counters().abs().sum()) == 0, name
    finally:
        mr.set_launch_flags(prev)
    assert_logits_close(host(lg), oracle.router_gemv(x, w))
