"""Sort and stage-1 quant in one launch (decode batches): bitwise equal to
the separate sort and quant calls, and to the oracle."""

import numpy as np
import pytest

import oracle
from decode_expert_routing_gb300 import inputs
from tests.gpu_util import check_sort, host, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mr():
    from decode_expert_routing_gb300 import build
    build.build()
    import decode_expert_routing_gb300 as m
    m.load_library()
    return m


@pytest.mark.parametrize("M,N,K,k,B,quant", [(1, 128, 6144, 8, 16, "mxfp8"), (65, 128, 6144, 8, 16, "mxfp4"),
                                             (300, 128, 6144, 8, 64, "mxfp8"), (1024, 128, 6144, 8, 16, "mxfp8"),
                                             (1024, 128, 6144, 8, 64, "mxfp4"), (512, 896, 3584, 16, 16, "mxfp8"),
                                             (256, 1024, 512, 32, 128, "mxfp4"), (7, 40, 64, 7, 1, "mxfp8")])
def test_sort_quant_equals_separate_calls_and_oracle(mr, M, N, K, k, B, quant):
    x = inputs.prefill_x(M, K)
    # ids: the oracle's gate on the oracle's logits (an input here, not a result under test)
    _, w = inputs.router_inputs(1, K, N, 4)
    ids, _ = oracle.route_topk(oracle.router_gemv(x, w), k)
    idd, xd = to_dev(ids), to_dev_bf16(x)
    st, ex, nt, q, s = mr.moe_sort_quant(idd, xd, N, B, quant)
    st2, ex2, nt2 = mr.moe_sort(idd, N, B)
    q2, s2 = (mr.mxfp4_quant if quant == "mxfp4" else mr.mxfp8_quant)(xd)
    for a, b in ((st, st2), (ex, ex2), (nt, nt2), (q, q2), (s, s2)):
        assert np.array_equal(host(a), host(b))
    check_sort(ids, N, B, host(st), host(ex), host(nt))
    wq, ws = (oracle.mxfp4_quant if quant == "mxfp4" else oracle.mxfp8_quant)(x)
    assert np.array_equal(host(q), wq) and np.array_equal(host(s), ws)


def test_sort_quant_limits(mr):
    x = to_dev_bf16(inputs.prefill_x(1025, 512))
    ids = to_dev(np.zeros((1025, 8), dtype=np.int32))
    with pytest.raises(mr.MoeRouteUnsupported):
        mr.moe_sort_quant(ids, x, 128, 16)
