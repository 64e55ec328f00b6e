"""The router GEMV alone above 64 token rows (the tensor-core kernel: staged
tensor copies, MMAs into tensor memory, split-K over a cluster) against the
oracle, over the shapes its plan covers: ragged row counts on both sides of
the 64/128-row cluster switch, expert counts that leave half a 16-wide MMA
column block, K slices that end inside a 64-wide stage, strided and offset x,
and integer inputs whose logits are exact in any summation order."""

import numpy as np
import pytest

import oracle
from decode_expert_routing_gb300 import inputs

from gpu_util import assert_logits_close, host, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mr():
    from decode_expert_routing_gb300 import build
    build.build()
    import decode_expert_routing_gb300 as m
    m.load_library()
    return m


def _run(mr, x, w, ldx_pad=0, row_off=0):
    """router_gemv on x (optionally inside a wider, row-offset buffer)."""
    M, K = x.shape
    if ldx_pad or row_off:
        buf = np.zeros((M + row_off, K + ldx_pad), np.uint16)
        buf[row_off:, :K] = x
        xd = to_dev_bf16(buf)[row_off:, :K]
    else:
        xd = to_dev_bf16(x)
    return host(mr.router_gemv(xd, to_dev_bf16(w)))


@pytest.mark.parametrize("M", [65, 100, 128, 129, 200, 256, 300, 448, 449, 511, 512])
def test_rows_past_64_match_oracle(mr, M):
    x, w = inputs.router_inputs(M, 6144, 128, 7)
    g1 = _run(mr, x, w)
    assert_logits_close(g1, oracle.router_gemv(x, w))
    g2 = _run(mr, x, w)
    assert np.array_equal(g1.view(np.uint32), g2.view(np.uint32)), "not deterministic"


@pytest.mark.parametrize("N", [8, 40, 64, 120, 128])
@pytest.mark.parametrize("M", [100, 512])
def test_expert_counts(mr, N, M):
    """N not a multiple of 16 leaves the MMA's last column block half empty."""
    x, w = inputs.router_inputs(M, 6144, N, 7)
    assert_logits_close(_run(mr, x, w), oracle.router_gemv(x, w))


@pytest.mark.parametrize("K", [512, 1024, 3584, 7168])
@pytest.mark.parametrize("M", [80, 512])
def test_hidden_sizes(mr, K, M):
    """K = 512: one stage, two k-steps, receive buffers after the weight
    stages; 3584: the last stage half used; 7168: seven stages."""
    x, w = inputs.router_inputs(M, K, 128, 7)
    assert_logits_close(_run(mr, x, w), oracle.router_gemv(x, w))


@pytest.mark.parametrize("M", [100, 512])
def test_strided_and_offset_x(mr, M):
    x, w = inputs.router_inputs(M, 6144, 128, 21)
    ref = oracle.router_gemv(x, w)
    assert_logits_close(_run(mr, x, w, ldx_pad=64), ref)
    assert_logits_close(_run(mr, x, w, row_off=3), ref)


@pytest.mark.parametrize("M", [65, 300, 512])
def test_integer_inputs_exact(mr, M):
    """Small-integer x and W: every partial sum is an integer below 2^24,
    exact in fp32 in any order, so the logits equal the oracle's bit for bit
    (a misplaced row, column or k-step changes some logit)."""
    rng = np.random.default_rng(1000 + M)
    K, N = 6144, 128
    xf = rng.integers(-2, 3, size=(M, K)).astype(np.float64)
    wf = rng.integers(-2, 3, size=(N, K)).astype(np.float64)
    x, w = inputs.f64_to_bf16_bits(xf), inputs.f64_to_bf16_bits(wf)
    g = _run(mr, x, w)
    ref = oracle.router_gemv(x, w)
    assert np.array_equal(g.astype(np.float64), ref)


def test_tied_rows_bitwise(mr):
    x, w = inputs.router_inputs(512, 6144, 128, 5)
    w = inputs.tied_gate(w)
    for M in (65, 300, 512):
        g = _run(mr, x[:M], w).view(np.uint32)
        assert np.array_equal(g[:, 10], g[:, 11]) and np.array_equal(g[:, 50], g[:, 51])


def test_bounded_wait_runs_out_and_reports(mr):
    """With the test hook each owner expects 16 bytes that never come: its
    wait ends at the limit, the device flag is set, and the next call is
    correct."""
    import torch
    x, w = inputs.router_inputs(200, 6144, 128, 7)
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    torch.cuda.synchronize()
    assert mr.device_error() == mr.MR_OK
    flags = mr.get_launch_flags()
    mr.set_wait_limit_ns(20_000_000)
    mr.set_launch_flags(flags | mr.LAUNCH_TEST_STALL)
    try:
        mr.router_gemv(xd, wd)
        torch.cuda.synchronize()
    finally:
        mr.set_launch_flags(flags)
        mr.set_wait_limit_ns(1_000_000_000)
    assert mr.device_error(clear=True) == mr.MR_ERR_TIMEOUT
    assert mr.device_error() == mr.MR_OK
    assert_logits_close(host(mr.router_gemv(xd, wd)), oracle.router_gemv(x, w))
    torch.cuda.synchronize()
    assert mr.device_error() == mr.MR_OK
