"""MXFP4 stage-1 activations: the standalone quantiser and the one-launch
route with quant="mxfp4" against the oracle, byte for byte, and the route's
general entry point (mr_moe_route) against the specific ones."""

import numpy as np
import pytest

import oracle
from decode_expert_routing_gb300 import inputs
from tests.gpu_util import host, to_dev, to_dev_bf16

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


def _check_q4(mr, x, pad=0):
    M, K = x.shape
    xp = np.zeros((M, K + pad), dtype=np.uint16)
    xp[:, :K] = x
    xd = to_dev_bf16(xp)[:, :K]
    q, s = mr.mxfp4_quant(xd)
    wq, ws = oracle.mxfp4_quant(x)
    qh, sh = host(q), host(s)
    bad = np.argwhere(qh != wq)
    assert bad.size == 0, f"q differs at {bad[:4].tolist()}: {qh[tuple(bad[0])]:#04x} vs {wq[tuple(bad[0])]:#04x}"
    assert np.array_equal(sh, ws)


@pytest.mark.parametrize("M,K,pad", [(1, 32, 0), (3, 6144, 0), (64, 6144, 8), (33, 3584, 64), (257, 512, 0)])
def test_mxfp4_quant_equals_oracle(mr, M, K, pad):
    x, _ = inputs.router_inputs(M, K, 8, 2)
    _check_q4(mr, x, pad)


def test_mxfp4_quant_edge_blocks(mr):
    _check_q4(mr, inputs.quant_edge_x(64, 6144))


def test_mxfp4_quant_every_bf16_pattern(mr):
    # all 65,280 finite bf16 patterns, in order (blocks of neighbouring
    # magnitudes: scales from the clamped lowest up to the largest) and in a
    # seeded shuffle (blocks mixing magnitudes: saturation and flush to zero)
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    b = b[(b & 0x7F80) != 0x7F80]
    assert b.size == 34 * 1920
    _check_q4(mr, b.reshape(34, 1920))
    perm = inputs.fisher_yates(b.size, inputs.stream_key(4, 77))
    _check_q4(mr, b[perm].reshape(34, 1920))


def test_mxfp4_prefill_rows(mr):
    x = inputs.prefill_x(4096, 6144)
    _check_q4(mr, x)


@pytest.mark.parametrize("M,norm", [(1, False), (8, False), (16, True), (32, False), (64, True)])
def test_route_mxfp4_equals_standalone_and_oracle(mr, M, norm):
    K, N, topk, block = 6144, 128, 8, 16
    _, w = inputs.router_inputs(1, K, N, 2)
    wd = to_dev_bf16(w)
    if norm:
        s, r, g = inputs.norm_inputs(M, K)
        xd, rd, gd = to_dev_bf16(s), to_dev(r), to_dev_bf16(g)
        xn = oracle.norm_apply(s, r, g, "gemma")
    else:
        x, _ = inputs.router_inputs(M, K, N, 2)
        xd, rd, gd = to_dev_bf16(x), None, None
        xn = x
    scratch = mr.Scratch(M, N, K, topk)
    f4 = mr.moe_route(xd, wd, topk, block, quant="mxfp4", rstd=rd, norm_weight=gd, scratch=scratch)
    f8 = mr.moe_route(xd, wd, topk, block, quant="mxfp8", rstd=rd, norm_weight=gd, scratch=scratch)
    f0 = mr.moe_route(xd, wd, topk, block, quant=None, rstd=rd, norm_weight=gd, scratch=scratch)
    assert "q" not in f0
    for key in f0:   # the format changes nothing but q
        assert np.array_equal(_bits(f4[key]), _bits(f8[key])), key
        assert np.array_equal(_bits(f4[key]), _bits(f0[key])), key
    wq, ws = oracle.mxfp4_quant(xn)
    assert np.array_equal(host(f4["q"]), wq)
    assert np.array_equal(host(f4["scale"]), ws)
    q8, s8 = oracle.mxfp8_quant(xn)
    assert np.array_equal(host(f8["q"]), q8) and np.array_equal(host(f8["scale"]), s8)
    # the specific entry points are this one with MXFP8
    if norm:
        spec = mr.moe_route_sort_quant_norm(xd, rd, gd, wd, topk, block, "gemma", scratch=scratch)
    else:
        spec = mr.moe_route_sort_quant(xd, wd, topk, block, scratch=scratch)
    for key in spec:
        assert np.array_equal(_bits(spec[key]), _bits(f8[key])), key
    assert int(scratch.counters().abs().sum()) == 0


def test_prepared_route_equals_moe_route(mr):
    import torch
    M, K, N = 8, 6144, 128
    x, w = inputs.router_inputs(M, K, N, 2)
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    call = mr.PreparedRoute(xd, wd, 8, 16, quant="mxfp4")
    out = call()
    ref = mr.moe_route(xd, wd, 8, 16, quant="mxfp4")
    for key in ref:
        assert np.array_equal(_bits(out[key]), _bits(ref[key])), key
    # refill x in place and launch again on a raw stream handle
    x2, _ = inputs.router_inputs(M, K, N, 2, variant=1)
    xd.copy_(to_dev_bf16(x2))
    s = torch.cuda.Stream()
    call(s.cuda_stream)
    s.synchronize()
    ref2 = mr.moe_route(to_dev_bf16(x2), wd, 8, 16, quant="mxfp4")
    for key in ref2:
        assert np.array_equal(_bits(out[key]), _bits(ref2[key])), key
