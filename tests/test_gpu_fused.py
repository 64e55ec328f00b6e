"""The one-launch route (M <= 64): bitwise equal to the four-call chain, and
to the oracle where the oracle is exact; 1000 back-to-back launches on one
scratch buffer, every launch checked."""

import numpy as np
import pytest

import oracle
from decode_expert_routing_gb300 import inputs
from tests.gpu_util import (assert_logits_close, check_gate, check_quant, check_sort, host,
                            to_dev, to_dev_bf16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mr():
    from decode_expert_routing_gb300 import build
    build.build()
    import decode_expert_routing_gb300 as m
    m.load_library()
    return m


def _chain(mr, xd, wd, c, bias_d, scratch):
    logits = mr.router_gemv(xd, wd, scratch=scratch)
    ids, wts = mr.route_topk(logits, c["topk"], c["scoring"], bias_d)
    st, ex, nt = mr.moe_sort(ids, c["N"], c["block"], scratch=scratch)
    q, s = mr.mxfp8_quant(xd)
    return dict(logits=logits, topk_ids=ids, topk_weights=wts, sorted_token_ids=st, expert_ids=ex,
                num_tokens_post_padded=nt, q=q, scale=s)


def _bits(t):
    a = host(t)
    return a.view(np.uint32) if a.dtype == np.float32 else a


@pytest.mark.parametrize("cid,M", [(1, 1), (2, 2), (2, 4), (2, 8), (2, 16), (2, 32), (2, 64), (3, 1),
                                   (3, 8), (3, 16), (3, 32), (2, 3), (2, 11), (2, 17), (2, 47), (5, 64)])
def test_fused_equals_chain_and_oracle(mr, cid, M):
    c = inputs.CONFIGS[cid]
    x, w = inputs.router_inputs(M, c["K"], c["N"], cid)
    bias = inputs.selection_bias(c["N"]) if c["scoring"] == "sigmoid" else None
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    bd = None if bias is None else to_dev(bias)
    scratch = mr.Scratch(M, c["N"], c["K"], c["topk"])
    fused = mr.moe_route_sort_quant(xd, wd, c["topk"], c["block"], c["scoring"], bd, scratch=scratch)
    chain = _chain(mr, xd, wd, c, bd, scratch)
    lh = host(fused["logits"])
    # each side against the oracle first (on the GPU's own ids), then bit for bit
    check_sort(host(chain["topk_ids"]), c["N"], c["block"], host(chain["sorted_token_ids"]),
               host(chain["expert_ids"]), host(chain["num_tokens_post_padded"]))
    for key in chain:
        f, ch = _bits(fused[key]), _bits(chain[key])
        bad = np.flatnonzero(f.reshape(-1) != ch.reshape(-1))
        assert bad.size == 0, f"{key} differs from the chain at {bad[:6].tolist()}: {f.reshape(-1)[bad[:6]].tolist()} vs {ch.reshape(-1)[bad[:6]].tolist()}"
    assert int(scratch.counters().abs().sum()) == 0
    assert_logits_close(lh, oracle.router_gemv(x, w))
    check_gate(lh, host(fused["topk_ids"]), host(fused["topk_weights"]), c["topk"], c["scoring"], bias)
    check_sort(host(fused["topk_ids"]), c["N"], c["block"], host(fused["sorted_token_ids"]),
               host(fused["expert_ids"]), host(fused["num_tokens_post_padded"]))
    check_quant(x, host(fused["q"]), host(fused["scale"]))


@pytest.mark.parametrize("K,N", [(512, 64), (2048, 128), (3072, 128), (4096, 128), (7168, 128), (6144, 256)])
@pytest.mark.parametrize("M", [1, 8, 16, 40])
def test_every_k_step_count(mr, K, N, M):
    """The route kernel is compiled for 6 and 7 k steps per k-part (K =
    3072 / 6144 and 7168 on 16 CTAs) and for a run-time count otherwise (K =
    512: 1, 2048: 4, 4096: 8): each against the oracle, and the GEMV alone
    bitwise equal to the route's logits."""
    x, w = inputs.router_inputs(M, K, N, 2)
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    scratch = mr.Scratch(M, N, K, 8)
    fused = mr.moe_route_sort_quant(xd, wd, 8, 16, scratch=scratch)
    alone = mr.router_gemv(xd, wd, scratch=scratch)
    lh = host(fused["logits"])
    assert np.array_equal(lh.view(np.uint32), host(alone).view(np.uint32))
    assert_logits_close(lh, oracle.router_gemv(x, w))
    ids, _ = check_gate(lh, host(fused["topk_ids"]), host(fused["topk_weights"]), 8, "softmax")
    check_sort(ids, N, 16, host(fused["sorted_token_ids"]), host(fused["expert_ids"]),
               host(fused["num_tokens_post_padded"]))
    check_quant(x, host(fused["q"]), host(fused["scale"]))
    assert int(scratch.counters().abs().sum()) == 0


def test_fused_without_quant(mr):
    x, w = inputs.router_inputs(4, 6144, 128, 2)
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    out = mr.moe_route_sort_quant(xd, wd, 8, 16, quant=False)
    assert "q" not in out
    check_gate(host(out["logits"]), host(out["topk_ids"]), host(out["topk_weights"]), 8, "softmax")


@pytest.mark.parametrize("M,chain,pdl", [(2, "fused", 0), (4, "fused", 0), (8, "fused", 0), (16, "fused", 0),
                                         (32, "fused", 0), (64, "fused", 0), (32, "four calls", 0),
                                         (64, "four calls", 0), (4, "fused", 1), (17, "fused", 1),
                                         (64, "fused", 1), (64, "four calls", 1)])
def test_1000_launches_reuse_one_scratch(mr, M, chain, pdl):
    """Config 2: 1000 back-to-back launches on one scratch/counter buffer
    (the one-launch route, and the four separate calls), in plain stream
    order and with programmatic dependent launch (each kernel starting while
    the previous one runs); every launch's outputs land in a ring and each is
    checked against the reference outputs of its input variant."""
    import torch
    flags = mr.get_launch_flags()
    mr.set_launch_flags(mr.LAUNCH_PDL if pdl else 0)
    try:
        _run_1000(mr, M, chain)
    finally:
        mr.set_launch_flags(flags)
    assert mr.device_error() == mr.MR_OK


def _run_1000(mr, M, chain):
    import torch
    c = inputs.CONFIGS[2]
    K, N, k, B = c["K"], c["N"], c["topk"], c["block"]
    nvar, L = 4, 1000
    xs, ws = zip(*[inputs.router_inputs(M, K, N, 2, variant=v) for v in range(nvar)])
    xds = [to_dev_bf16(a) for a in xs]
    wds = [to_dev_bf16(a) for a in ws]
    scratch = mr.Scratch(M, N, K, k)
    cap = mr.sort_capacity(M, k, N, B)
    dev = xds[0].device
    ring = dict(
        logits=torch.empty((L, M, N), dtype=torch.float32, device=dev),
        topk_ids=torch.empty((L, M, k), dtype=torch.int32, device=dev),
        topk_weights=torch.empty((L, M, k), dtype=torch.float32, device=dev),
        sorted_token_ids=torch.empty((L, cap), dtype=torch.int32, device=dev),
        expert_ids=torch.empty((L, cap // B), dtype=torch.int32, device=dev),
        num_tokens_post_padded=torch.empty((L, 1), dtype=torch.int32, device=dev),
        q=torch.empty((L, M, K), dtype=torch.uint8, device=dev),
        scale=torch.empty((L, M, K // 32), dtype=torch.uint8, device=dev),
    )
    for i in range(L):
        v = i % nvar
        out = {key: t[i] for key, t in ring.items()}
        if chain == "fused":
            mr.moe_route_sort_quant(xds[v], wds[v], k, B, out=out, scratch=scratch)
        else:
            mr.router_gemv(xds[v], wds[v], out=out["logits"], scratch=scratch)
            mr.route_topk(out["logits"], k, ids=out["topk_ids"], weights=out["topk_weights"])
            mr.moe_sort(out["topk_ids"], N, B, scratch=scratch,
                        out=(out["sorted_token_ids"], out["expert_ids"], out["num_tokens_post_padded"]))
            mr.mxfp8_quant(xds[v], out=(out["q"], out["scale"]))
    torch.cuda.synchronize()
    assert int(scratch.counters().abs().sum()) == 0
    for v in range(nvar):
        first = {key: t[v] for key, t in ring.items()}
        for key, t in ring.items():
            tb = t.view(torch.int32) if t.dtype == torch.float32 else t
            same = (tb[v::nvar] == tb[v].unsqueeze(0)).reshape(tb[v::nvar].shape[0], -1).all(1)
            assert bool(same.all()), f"{key}: launch {v + nvar * int((~same).nonzero()[0])} differs"
        lh = host(first["logits"])
        assert_logits_close(lh, oracle.router_gemv(xs[v], ws[v]))
        check_gate(lh, host(first["topk_ids"]), host(first["topk_weights"]), k, "softmax")
        check_sort(host(first["topk_ids"]), N, B, host(first["sorted_token_ids"]),
                   host(first["expert_ids"]), host(first["num_tokens_post_padded"]))
        check_quant(xs[v], host(first["q"]), host(first["scale"]))


def test_bounded_wait_runs_out_and_reports(mr):
    """The cluster kernels' waits for bytes from other CTAs are bounded: with
    the test hook every receiving CTA expects 16 bytes that never come, so
    each wait ends at the limit, the device flag is set, and the context
    stays usable (a normal call afterwards is exact)."""
    import torch
    c = inputs.CONFIGS[2]
    x, w = inputs.router_inputs(4, c["K"], c["N"], 2)
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    torch.cuda.synchronize()
    assert mr.device_error() == mr.MR_OK  # no earlier call ran out
    flags = mr.get_launch_flags()
    mr.set_wait_limit_ns(20_000_000)
    mr.set_launch_flags(flags | mr.LAUNCH_TEST_STALL)
    try:
        mr.moe_route_sort_quant(xd, wd, c["topk"], c["block"])
        mr.router_gemv(xd, wd)
        torch.cuda.synchronize()
    finally:
        mr.set_launch_flags(flags)
        mr.set_wait_limit_ns(1_000_000_000)
    assert mr.device_error(clear=True) == mr.MR_ERR_TIMEOUT
    assert mr.device_error() == mr.MR_OK
    out = mr.moe_route_sort_quant(xd, wd, c["topk"], c["block"])
    lh = host(out["logits"])
    assert_logits_close(lh, oracle.router_gemv(x, w))
    check_gate(lh, host(out["topk_ids"]), host(out["topk_weights"]), c["topk"], c["scoring"], None)
    check_sort(host(out["topk_ids"]), c["N"], c["block"], host(out["sorted_token_ids"]),
               host(out["expert_ids"]), host(out["num_tokens_post_padded"]))
    torch.cuda.synchronize()
    assert mr.device_error() == mr.MR_OK
