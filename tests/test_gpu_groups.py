"""Routes over many experts split them into groups, one cluster per group
(per 16 tokens), and merge the groups' top-k candidates in the CTA that
finishes last.  Every output must equal the four-call chain bit for bit, the
unsplit one-launch route (a scratch too small for the candidates) bit for bit,
and the oracle (logits within tolerance; gate, sort and quant exact)."""

import numpy as np
import pytest
import torch

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


def _bits(t):
    a = host(t)
    return a.view(np.uint32) if a.dtype == np.float32 else a


CASES = [  # M, N, K, topk, scoring, renormalize, block
    (1, 896, 3584, 16, "sigmoid", True, 16),
    (8, 896, 3584, 16, "sigmoid", True, 16),
    (16, 896, 3584, 16, "sigmoid", False, 16),
    (32, 896, 3584, 16, "sigmoid", True, 16),
    (64, 896, 3584, 16, "sigmoid", True, 64),
    (16, 1024, 6144, 32, "softmax", True, 16),
    (11, 1024, 6144, 32, "softmax", False, 32),
    (17, 512, 6144, 8, "softmax", True, 16),
    (3, 512, 512, 8, "softmax", False, 16),
    (47, 640, 1024, 8, "softmax", True, 128),
]


@pytest.mark.parametrize("M,N,K,k,scoring,renorm,B", CASES)
def test_groups_equal_chain_unsplit_and_oracle(mr, M, N, K, k, scoring, renorm, B):
    x, w = inputs.router_inputs(M, K, N, 3)
    bias = inputs.selection_bias(N) if scoring == "sigmoid" else None
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    bd = None if bias is None else to_dev(bias)
    scratch = mr.Scratch(M, N, K, k)
    small = mr.Scratch(min(M, 16), 8, K, 1)          # no room for group candidates
    split = mr.moe_route_sort_quant(xd, wd, k, B, scoring, bd, renorm, scratch=scratch)
    if M <= 16:
        unsplit = mr.moe_route_sort_quant(xd, wd, k, B, scoring, bd, renorm, scratch=small)
    logits = mr.router_gemv(xd, wd, scratch=scratch)
    ids, wts = mr.route_topk(logits, k, scoring, bd, renorm)
    st, ex, nt = mr.moe_sort(ids, N, B, scratch=scratch)
    q, s = mr.mxfp8_quant(xd)
    chain = dict(logits=logits, topk_ids=ids, topk_weights=wts, sorted_token_ids=st, expert_ids=ex,
                 num_tokens_post_padded=nt, q=q, scale=s)
    for key in chain:
        f, c = _bits(split[key]), _bits(chain[key])
        bad = np.flatnonzero(f.reshape(-1) != c.reshape(-1))
        assert bad.size == 0, f"{key} differs from the chain at {bad[:6].tolist()}"
        if M <= 16:
            assert np.array_equal(_bits(unsplit[key]), f), f"{key}: split and unsplit differ"
    assert int(scratch.counters().abs().sum()) == 0
    lh = host(split["logits"])
    assert_logits_close(lh, oracle.router_gemv(x, w))
    check_gate(lh, host(split["topk_ids"]), host(split["topk_weights"]), k, scoring, bias, renorm)
    check_sort(host(split["topk_ids"]), N, B, host(split["sorted_token_ids"]), host(split["expert_ids"]),
               host(split["num_tokens_post_padded"]))
    check_quant(x, host(split["q"]), host(split["scale"]))


@pytest.mark.parametrize("pdl", [0, 1])
def test_groups_300_launches_on_one_scratch(mr, pdl):
    M, N, K, k, B = 16, 896, 3584, 16, 16
    nvar, L = 3, 300
    xs, ws = zip(*[inputs.router_inputs(M, K, N, 3, variant=v) for v in range(nvar)])
    xds, wds = [to_dev_bf16(a) for a in xs], [to_dev_bf16(a) for a in ws]
    bd = to_dev(inputs.selection_bias(N))
    scratch = mr.Scratch(M, N, K, k)
    outs = [mr.alloc_route_outputs(M, N, K, k, B, xds[0].device) for _ in range(L)]
    mr.set_launch_flags(mr.LAUNCH_PDL if pdl else 0)
    try:
        for i in range(L):
            mr.moe_route_sort_quant(xds[i % nvar], wds[i % nvar], k, B, "sigmoid", bd, out=outs[i], scratch=scratch)
        torch.cuda.synchronize()
    finally:
        mr.set_launch_flags(0)
    assert int(scratch.counters().abs().sum()) == 0
    for i in range(nvar, L):
        for key in outs[i]:
            assert np.array_equal(_bits(outs[i][key]), _bits(outs[i % nvar][key])), (i, key)
    for v in range(nvar):
        lh = host(outs[v]["logits"])
        assert_logits_close(lh, oracle.router_gemv(xs[v], ws[v]))
        check_gate(lh, host(outs[v]["topk_ids"]), host(outs[v]["topk_weights"]), k, "sigmoid",
                   inputs.selection_bias(N))
