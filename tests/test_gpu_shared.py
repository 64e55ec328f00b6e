"""The shared expert's gate/up projection and SwiGLU (mr_shared_gate_up),
alone and fused into the one-launch route (mr_moe_route with shared_w13).

Tolerance, derived from the arithmetic: the kernel sums each 32-wide block
of a row in the MMA (products exact), scales it with one fused
multiply-add, accumulates at most 8 blocks per k-part, and the owner adds
the 32 (or 16) split-K partials: fewer than 2^6 roundings of 2^-24 relative
to the running sum, so |dh| <= 2^-18 * sum_k |x W|; 2^-16 is used.  Then
act = silu(g) * u moves by at most 1.1 |u| dg + |silu(g)| du (|silu'| <
1.1), the fp32 silu and product add a few 2^-24 relative, and both sides
round to bf16, which can part them by one bf16 spacing."""

import numpy as np
import pytest

import oracle
from decode_expert_routing_gb300 import inputs
from tests.gpu_util import check_gate, check_quant, check_sort, host, to_dev, to_dev_bf16, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mr():
    from decode_expert_routing_gb300 import build
    build.build()
    import decode_expert_routing_gb300 as m
    m.load_library()
    return m


def _bf16_vals(bits):
    return inputs.bf16_bits_to_f32(np.asarray(bits, np.uint16)).astype(np.float64)


def _dequant(codes, scale):
    table = np.array([oracle.e4m3_decode(c) for c in range(256)])
    return table[codes] * np.exp2(np.repeat(scale.astype(np.float64) - 127, 32, axis=1))


def assert_act_close(gpu_bits, x, codes, scale):
    ref_bits, h = oracle.shared_gate_up(x, codes, scale)
    I = ref_bits.shape[1]
    absw = np.abs(_dequant(codes, scale))
    mag = np.abs(_bf16_vals(x)) @ absw.T          # sum_k |x W| per (m, r)
    dh = mag * 2.0 ** -16
    g, u = h[:, :I], h[:, I:]
    with np.errstate(over="ignore"):  # exp(-g) = inf for very negative g: silu -> -0
        silu = g / (1 + np.exp(-g))
    ref, got = _bf16_vals(ref_bits), _bf16_vals(gpu_bits)
    ulp = np.maximum(np.abs(ref), np.abs(got)) * 2.0 ** -7
    bound = 1.1 * np.abs(u) * dh[:, :I] + np.abs(silu) * dh[:, I:] + 1e-6 * np.abs(ref) + ulp + 1e-30
    err = np.abs(got - ref)
    assert np.all(err <= bound), f"worst {np.max(err / bound):.3f} of the bound at {np.unravel_index(np.argmax(err / bound), err.shape)}"
    return np.mean(gpu_bits == ref_bits)


@pytest.mark.parametrize("M,K,I", [(1, 6144, 768), (4, 6144, 768), (8, 6144, 768), (16, 6144, 768),
                                   (3, 512, 64), (16, 3584, 256), (5, 6144, 1536)])
def test_shared_gate_up_matches_oracle(mr, M, K, I):
    x, _ = inputs.router_inputs(M, K, 8, 7)
    codes, scale = inputs.shared_expert_weights(I, K)
    out = mr.shared_gate_up(to_dev_bf16(x), to_dev(codes), to_dev(scale))
    same = assert_act_close(host(out.view(torch_mod().int16)).view(np.uint16), x, codes, scale)
    print(f"M={M} K={K} I={I}: {same:.4f} of the bf16 outputs equal the oracle's bits")


def test_shared_gate_up_is_deterministic_and_strided(mr):
    M, K, I = 8, 6144, 768
    xw, _ = inputs.router_inputs(M, 2 * K, 8, 7)
    codes, scale = inputs.shared_expert_weights(I, K)
    xs = to_dev_bf16(xw)[:, 128:128 + K]  # a row stride of 2K
    a = host(mr.shared_gate_up(xs, to_dev(codes), to_dev(scale)).view(torch_mod().int16))
    b = host(mr.shared_gate_up(xs.contiguous(), to_dev(codes), to_dev(scale)).view(torch_mod().int16))
    assert np.array_equal(a, b)
    assert_act_close(a.view(np.uint16), np.ascontiguousarray(xw[:, 128:128 + K]), codes, scale)


@pytest.mark.parametrize("case", ["some slices", "every slice"])
def test_shared_gate_up_values_outside_f16(mr, case):
    """A CTA whose x slice holds a value that f16 does not carry exactly
    (at or above 2^16, or below 2^-17 and not zero) runs the bf16 MMAs; the
    others the f16 ones.  Both against the oracle: one large and one tiny
    value in two K slices, or x scaled by 2^17 so that every slice holds
    values past f16's range."""
    M, K, I = 4, 6144, 768
    x, _ = inputs.router_inputs(M, K, 8, 7)
    xf = inputs.bf16_bits_to_f32(x).astype(np.float64)
    if case == "some slices":
        xf[0, 5] = 3.0e5       # slice 0 (K / 16 = 384 columns a slice)
        xf[1, 3000] = 1.0e-6   # slice 7
        xf[2, 3001] = -2.0e-6
    else:
        xf *= 2.0 ** 17
    xb = inputs.f64_to_bf16_bits(xf)
    codes, scale = inputs.shared_expert_weights(I, K)
    out = mr.shared_gate_up(to_dev_bf16(xb), to_dev(codes), to_dev(scale))
    assert_act_close(host(out.view(torch_mod().int16)).view(np.uint16), xb, codes, scale)

@pytest.mark.parametrize("v", [2.0 ** -17, -(2.0 ** -17) * 1.5, 65280.0, -65280.0, 2.0 ** -18, 65536.0])
def test_shared_gate_up_f16_range_edges(mr, v):
    """Values at the edges of f16's exact range in one slice: 2^-17 (f16
    subnormal spacing 2^-24 still carries the bf16's last bit), 65280 (the
    largest bf16 below 2^16) stay on the f16 MMAs; 2^-18 (a bit lost) and
    2^16 (past f16's largest value) send the slice to the bf16 MMAs.  Either
    way the result matches the oracle."""
    M, K, I = 2, 6144, 768
    x, _ = inputs.router_inputs(M, K, 8, 7)
    xf = inputs.bf16_bits_to_f32(x).astype(np.float64)
    xf[1, 4000] = v
    xb = inputs.f64_to_bf16_bits(xf)
    assert inputs.bf16_bits_to_f32(xb)[1, 4000] == np.float32(v)
    codes, scale = inputs.shared_expert_weights(I, K)
    out = mr.shared_gate_up(to_dev_bf16(xb), to_dev(codes), to_dev(scale))
    assert_act_close(host(out.view(torch_mod().int16)).view(np.uint16), xb, codes, scale)

def _route_outputs_equal(a, b):
    for name in ("logits", "topk_ids", "topk_weights", "sorted_token_ids", "expert_ids",
                 "num_tokens_post_padded", "q", "scale"):
        assert np.array_equal(host(a[name]).view(np.uint8), host(b[name]).view(np.uint8)), name


@pytest.mark.parametrize("M", [1, 2, 8, 16])
def test_route_with_shared_expert_in_one_launch(mr, M):
    """The route and the shared expert in one launch: the route's outputs
    are the same bits as without it, the shared expert's those of
    mr_shared_gate_up, and both match the oracle."""
    torch = torch_mod()
    K, N, k, B, I = 6144, 128, 8, 16, 768
    x, w = inputs.router_inputs(M, K, N, 2)
    codes, scale = inputs.shared_expert_weights(I, K)
    xd, wd, cd, sd = to_dev_bf16(x), to_dev_bf16(w), to_dev(codes), to_dev(scale)
    fused = mr.moe_route(xd, wd, k, B, shared=(cd, sd))
    plain = mr.moe_route(xd, wd, k, B)
    alone = mr.shared_gate_up(xd, cd, sd)
    torch.cuda.synchronize()
    _route_outputs_equal(fused, plain)
    fa = host(fused["shared_act"].view(torch.int16))
    assert np.array_equal(fa, host(alone.view(torch.int16)))
    assert_act_close(fa.view(np.uint16), x, codes, scale)
    lh = host(fused["logits"])
    ids, _ = check_gate(lh, host(fused["topk_ids"]), host(fused["topk_weights"]), k, "softmax")
    check_sort(ids, N, B, host(fused["sorted_token_ids"]), host(fused["expert_ids"]),
               host(fused["num_tokens_post_padded"]))
    check_quant(x, host(fused["q"]), host(fused["scale"]))


def test_route_with_shared_expert_on_the_norm_scale_and_groups(mr):
    """On the norm's scale the shared expert reads the norm's output too;
    with 896 experts the route runs expert groups beside the shared clusters."""
    torch = torch_mod()
    K, N, k, B, I = 6144, 128, 8, 16, 768
    sres, rstd, g = inputs.norm_inputs(4, K)
    _, w = inputs.router_inputs(4, K, N, 2)
    codes, scale = inputs.shared_expert_weights(I, K)
    sd, rd, gd = to_dev_bf16(sres), to_dev(rstd), to_dev_bf16(g)
    cd, scd = to_dev(codes), to_dev(scale)
    fused = mr.moe_route(sd, to_dev_bf16(w), k, B, rstd=rd, norm_weight=gd, shared=(cd, scd))
    xn = mr.norm_apply(sd, rd, gd, "gemma")
    alone = mr.shared_gate_up(xn, cd, scd)
    torch.cuda.synchronize()
    assert np.array_equal(host(fused["shared_act"].view(torch.int16)), host(alone.view(torch.int16)))
    K3, N3, k3 = 3584, 896, 16
    x3, w3 = inputs.router_inputs(8, K3, N3, 3)
    c3, s3 = inputs.shared_expert_weights(256, K3)
    bias = to_dev(inputs.selection_bias(N3))
    x3d, w3d = to_dev_bf16(x3), to_dev_bf16(w3)
    scr = mr.Scratch(8, N3, K3, k3)
    f3 = mr.moe_route(x3d, w3d, k3, B, "sigmoid", bias, shared=(to_dev(c3), to_dev(s3)), scratch=scr)
    p3 = mr.moe_route(x3d, w3d, k3, B, "sigmoid", bias, scratch=scr)
    torch.cuda.synchronize()
    _route_outputs_equal(f3, p3)
    assert_act_close(host(f3["shared_act"].view(torch.int16)).view(np.uint16), x3, c3, s3)


def test_route_with_shared_expert_back_to_back_pdl(mr):
    """Programmatic dependent launch: consecutive fused launches on one
    stream, each checked."""
    torch = torch_mod()
    K, N, k, B, I = 6144, 128, 8, 16, 768
    codes, scale = inputs.shared_expert_weights(I, K)
    cd, sd = to_dev(codes), to_dev(scale)
    xs = [inputs.router_inputs(8, K, N, 2, variant=v) for v in range(3)]
    prev = mr.get_launch_flags()
    mr.set_launch_flags(prev | mr.LAUNCH_PDL)
    try:
        outs = [mr.moe_route(to_dev_bf16(x), to_dev_bf16(w), k, B, shared=(cd, sd)) for (x, w) in xs * 2]
        torch.cuda.synchronize()
    finally:
        mr.set_launch_flags(prev)
    assert mr.device_error() == mr.MR_OK
    for (x, w), o in zip(xs * 2, outs):
        assert_act_close(host(o["shared_act"].view(torch.int16)).view(np.uint16), x, codes, scale)
