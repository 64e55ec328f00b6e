"""The route on the norm's scale: the router takes the un-normalised residual
rows, each token's rstd and the norm weight, and forms its input in the
kernel.  The written-out input equals the oracle's bit for bit; the one
launch equals the written-out input followed by the one-launch route, bit
for bit; and against the oracle the route meets the same bars as the plain
route (logits within tolerance, gate / sort / quant exact)."""

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
    return a.view(np.uint32) if a.dtype == np.float32 else a.view(np.uint16) if a.dtype == np.int16 else a


def _bf16_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("M,K,kind,pad", [(1, 6144, "gemma", 0), (7, 6144, "rms", 0), (64, 6144, "gemma", 0),
                                          (33, 3584, "rms", 64), (300, 512, "gemma", 8), (5, 8, "gemma", 0)])
def test_norm_apply_equals_oracle(mr, M, K, kind, pad):
    s, r, g = inputs.norm_inputs(M, K)
    if kind == "rms":
        g = inputs.f64_to_bf16_bits(1.0 + inputs.bf16_bits_to_f32(g).astype(np.float64))
    want = oracle.norm_apply(s, r, g, kind)
    sp = np.zeros((M, K + pad), dtype=np.uint16)
    sp[:, :K] = s
    sd = to_dev_bf16(sp)[:, :K]                    # row pitch K + pad
    got = mr.norm_apply(sd, to_dev(r), to_dev_bf16(g), kind)
    assert np.array_equal(_bf16_bits(got), want)


def test_norm_apply_subnormal_and_tie_cases(mr):
    # rows whose products land on bf16 ties and among bf16 subnormals
    xv = np.array([[1.0, -1.0, 1.0 + 2 ** -7, 3.0, 1.0, 5.0, -3.0, 1.0]])
    rv = np.array([1 + 2 ** -8], dtype=np.float32)
    x = inputs.f64_to_bf16_bits(xv)
    g = np.full(8, 0x3F80, dtype=np.uint16)
    got = mr.norm_apply(to_dev_bf16(x), to_dev(rv), to_dev_bf16(g), "rms")
    assert np.array_equal(_bf16_bits(got), oracle.norm_apply(x, rv, g, "rms"))
    rv2 = np.array([2.0 ** -134], dtype=np.float32)
    got = mr.norm_apply(to_dev_bf16(x), to_dev(rv2), to_dev_bf16(g), "rms")
    assert np.array_equal(_bf16_bits(got), oracle.norm_apply(x, rv2, g, "rms"))


@pytest.mark.parametrize("M,kind", [(1, "gemma"), (2, "gemma"), (4, "rms"), (8, "gemma"), (16, "gemma"),
                                    (17, "rms"), (32, "gemma"), (47, "gemma"), (64, "gemma")])
def test_route_norm_equals_chain_and_oracle(mr, M, kind):
    c = inputs.CONFIGS[6]
    K, N, topk, block = c["K"], c["N"], c["topk"], c["block"]
    s, r, g = inputs.norm_inputs(M, K)
    if kind == "rms":
        g = inputs.f64_to_bf16_bits(1.0 + inputs.bf16_bits_to_f32(g).astype(np.float64))
    _, w = inputs.router_inputs(1, K, N, 6)
    sd, rd, gd, wd = to_dev_bf16(s), to_dev(r), to_dev_bf16(g), to_dev_bf16(w)
    scratch = mr.Scratch(M, N, K, topk)
    fused = mr.moe_route_sort_quant_norm(sd, rd, gd, wd, topk, block, kind, scratch=scratch)
    xn_d = mr.norm_apply(sd, rd, gd, kind)
    chain = mr.moe_route_sort_quant(xn_d, wd, topk, block, scratch=scratch)
    for key in chain:
        f, ch = _bits(fused[key]), _bits(chain[key])
        bad = np.flatnonzero(f.reshape(-1) != ch.reshape(-1))
        assert bad.size == 0, f"{key} differs from the written-out chain at {bad[:6].tolist()}"
    assert int(scratch.counters().abs().sum()) == 0
    xn = oracle.norm_apply(s, r, g, kind)
    assert np.array_equal(_bf16_bits(xn_d), xn)
    lh = host(fused["logits"])
    assert_logits_close(lh, oracle.router_gemv(xn, w))
    check_gate(lh, host(fused["topk_ids"]), host(fused["topk_weights"]), topk, "softmax")
    check_sort(host(fused["topk_ids"]), N, block, host(fused["sorted_token_ids"]), host(fused["expert_ids"]),
               host(fused["num_tokens_post_padded"]))
    check_quant(xn, host(fused["q"]), host(fused["scale"]))


def test_route_norm_large_expert_sigmoid(mr):
    # 896 experts, hidden 3584, sigmoid + selection bias, top-16, 8 tokens
    c = inputs.CONFIGS[3]
    M, K, N, topk, block = 8, c["K"], c["N"], c["topk"], c["block"]
    s, r, g = inputs.norm_inputs(M, K, config_id=3)
    _, w = inputs.router_inputs(1, K, N, 3)
    bias = inputs.selection_bias(N)
    sd, rd, gd, wd, bd = to_dev_bf16(s), to_dev(r), to_dev_bf16(g), to_dev_bf16(w), to_dev(bias)
    fused = mr.moe_route_sort_quant_norm(sd, rd, gd, wd, topk, block, "gemma", "sigmoid", bd)
    chain = mr.moe_route_sort_quant(mr.norm_apply(sd, rd, gd, "gemma"), wd, topk, block, "sigmoid", bd)
    for key in chain:
        assert np.array_equal(_bits(fused[key]), _bits(chain[key])), key
    xn = oracle.norm_apply(s, r, g, "gemma")
    lh = host(fused["logits"])
    assert_logits_close(lh, oracle.router_gemv(xn, w))
    check_gate(lh, host(fused["topk_ids"]), host(fused["topk_weights"]), topk, "sigmoid", bias)
    check_quant(xn, host(fused["q"]), host(fused["scale"]))


def test_route_norm_identity_scale_equals_plain_route(mr):
    # rstd = 1 and a Gemma weight of 0 leave the rows as they are: the route
    # on the norm's scale equals the plain route on the same rows
    M, K, N = 16, 6144, 128
    x, w = inputs.router_inputs(M, K, N, 2)
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    ones = torch.ones(M, dtype=torch.float32, device="cuda")
    zeros = torch.zeros(K, dtype=torch.bfloat16, device="cuda")
    a = mr.moe_route_sort_quant_norm(xd, ones, zeros, wd, 8, 16, "gemma")
    b = mr.moe_route_sort_quant(xd, wd, 8, 16)
    for key in b:
        assert np.array_equal(_bits(a[key]), _bits(b[key])), key
