"""The allocation-free router GEMV (mr_router_gemv_noalloc).

Some callers cannot allocate device memory or hand this library a scratch
buffer (for example plugins whose host framework owns all device memory).
This entry point uses a fixed-size scratch array that the library itself
declares.  Here it is called through the C ABI, twice in a row and in longer
back-to-back runs, and each result is compared with the oracle's fp64 GEMV
and with mr_router_gemv's output, within the logit tolerance of the other
GPU tests.  This file is collected last so that a run stopping at the first
failure has already run everything else; it also passes on its own in a
fresh process (the first call does the per-device set-up).
"""

import ctypes

import numpy as np
import pytest

import oracle
from decode_expert_routing_gb300 import inputs
from tests.gpu_util import assert_logits_close, host, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mr():
    from decode_expert_routing_gb300 import build
    build.build()
    import decode_expert_routing_gb300 as m
    m.load_library()
    return m


def _call(mr, xd, wd, out, M, N, K, stream):
    lib = mr.load_library()
    return lib.mr_router_gemv_noalloc(ctypes.c_void_p(xd.data_ptr()), K, ctypes.c_void_p(wd.data_ptr()),
                                      ctypes.c_void_p(out.data_ptr()), M, N, K, stream)


@pytest.mark.parametrize("M,N,K", [(2, 128, 6144), (100, 128, 6144), (512, 128, 6144), (16, 896, 3584)])
def test_noalloc_gemv_two_calls_match_oracle_and_router_gemv(mr, M, N, K):
    import torch
    x, w = inputs.router_inputs(M, K, N, 4)
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    want = oracle.router_gemv(x, w)
    ref = host(mr.router_gemv(xd, wd, scratch=mr.Scratch(M, N, K, 8)))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.float32, device=xd.device)
        st = _call(mr, xd, wd, out, M, N, K, stream)
        assert st == mr.MR_OK, mr.load_library().mr_status_string(st)
        torch.cuda.synchronize()
        assert_logits_close(host(out), want)
        assert_logits_close(host(out), ref)


def test_noalloc_gemv_allocates_nothing(mr):
    """After the set-up call, further calls leave the device's free memory
    unchanged (the library holds its array from load time on)."""
    import torch
    M, N, K = 64, 128, 6144
    x, w = inputs.router_inputs(M, K, N, 4)
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    out = torch.empty((M, N), dtype=torch.float32, device=xd.device)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert _call(mr, xd, wd, out, M, N, K, stream) == mr.MR_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(8):
        assert _call(mr, xd, wd, out, M, N, K, stream) == mr.MR_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert_logits_close(host(out), oracle.router_gemv(x, w))


@pytest.mark.parametrize("pdl", [False, True])
def test_noalloc_gemv_back_to_back_leaves_counters_zero(mr, pdl):
    """Several calls back to back on one stream (with and without
    programmatic dependent launch, where a call may start while the one
    before it finishes), each on its own input and output: every result
    matches the oracle, and a final call with the scratch check on finds the
    shared array's counters at zero."""
    import torch
    M, N, K = 100, 128, 6144
    xs = [inputs.router_inputs(M, K, N, 4, variant=v) for v in range(4)]
    xds = [(to_dev_bf16(x), to_dev_bf16(w)) for x, w in xs]
    outs = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in range(12)]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    prev = mr.get_launch_flags()
    mr.set_launch_flags(prev | (mr.LAUNCH_PDL if pdl else 0))
    try:
        for i, out in enumerate(outs):
            xd, wd = xds[i % 4]
            assert _call(mr, xd, wd, out, M, N, K, stream) == mr.MR_OK
        torch.cuda.synchronize()
        mr.set_launch_flags(prev | mr.LAUNCH_CHECK_SCRATCH)
        probe = torch.empty((M, N), dtype=torch.float32, device="cuda")
        assert _call(mr, xds[0][0], xds[0][1], probe, M, N, K, stream) == mr.MR_OK
        torch.cuda.synchronize()
    finally:
        mr.set_launch_flags(prev)
    for i, out in enumerate(outs):
        x, w = xs[i % 4]
        assert_logits_close(host(out), oracle.router_gemv(x, w))


def test_noalloc_refuses_problems_beyond_its_scratch(mr):
    lib = mr.load_library()
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: the size check refuses first
    # 64 splits x 512 rows x 1024 experts x 4 B = 128 MiB of partials > 8 MiB
    st = lib.mr_router_gemv_noalloc(fake, 16384, fake, fake, 512, 1024, 16384, None)
    assert st == mr.MR_ERR_UNSUPPORTED
