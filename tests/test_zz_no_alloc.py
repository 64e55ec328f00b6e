"""The allocation-free router GEMV (mr_router_gemv_noalloc).

Some callers cannot allocate device memory or hand this library a scratch
buffer (for example plugins whose host framework owns all device memory).
This entry point uses a fixed-size scratch array that the library itself
declares; here it is called through the C ABI twice in a row and each result
is compared with mr_router_gemv's output within the logit tolerance of the
other GPU tests.  This file is collected last so that a run stopping at the
first failure has already run everything else; it also passes on its own in
a fresh process (the first call does the per-device set-up).
"""

import ctypes

import numpy as np
import pytest

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


@pytest.mark.parametrize("M,N,K", [(2, 128, 6144), (100, 128, 6144), (512, 128, 6144), (16, 896, 3584)])
def test_noalloc_gemv_two_calls_match_router_gemv(mr, M, N, K):
    import torch
    lib = mr.load_library()
    x, w = inputs.router_inputs(M, K, N, 4)
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    ref = host(mr.router_gemv(xd, wd, scratch=mr.Scratch(M, N, K, 8)))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.float32, device=xd.device)
        st = lib.mr_router_gemv_noalloc(ctypes.c_void_p(xd.data_ptr()), K, ctypes.c_void_p(wd.data_ptr()),
                                        ctypes.c_void_p(out.data_ptr()), M, N, K, stream)
        assert st == mr.MR_OK, lib.mr_status_string(st)
        torch.cuda.synchronize()
        assert_logits_close(host(out), ref)


def test_noalloc_refuses_problems_beyond_its_scratch(mr):
    lib = mr.load_library()
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: the size check refuses first
    # 64 splits x 512 rows x 1024 experts x 4 B = 128 MiB of partials > 8 MiB
    st = lib.mr_router_gemv_noalloc(fake, 16384, fake, fake, 512, 1024, 16384, None)
    assert st == mr.MR_ERR_UNSUPPORTED
