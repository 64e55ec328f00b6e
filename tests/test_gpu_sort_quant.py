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
    x = to_dev_bf16(inputs.prefill_x(8193, 512))
    ids = to_dev(np.zeros((8193, 8), dtype=np.int32))
    with pytest.raises(mr.MoeRouteUnsupported):
        mr.moe_sort_quant(ids, x, 128, 16)


@pytest.mark.parametrize("quant", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("M,N,K,k,B", [(1, 128, 6144, 8, 16), (16, 128, 6144, 8, 16), (64, 128, 6144, 8, 16),
                                       (1024, 128, 6144, 8, 16), (200, 896, 3584, 16, 16), (9, 40, 64, 7, 4)])
def test_sort_quant_sorted_rows_match_oracle(mr, quant, M, N, K, k, B):
    """Stage-1 activations written in sorted order (the grouped GEMM's A
    rows): every row below num_tokens_post_padded equals the oracle's byte
    for byte (padding rows zero), rows past it are left untouched, and the
    sort outputs equal the token-order call's."""
    torch = __import__("torch")
    x = inputs.prefill_x(M, K)
    _, w = inputs.router_inputs(1, K, N, 4)
    ids, _ = oracle.route_topk(oracle.router_gemv(x, w), k)
    idd, xd = to_dev(ids), to_dev_bf16(x)
    cap = mr.sort_capacity(M, k, N, B)
    qk = K // 2 if quant == "mxfp4" else K
    out = (torch.empty(cap, dtype=torch.int32, device="cuda"), torch.empty(cap // B, dtype=torch.int32, device="cuda"),
           torch.empty(1, dtype=torch.int32, device="cuda"),
           torch.full((cap, qk), 0xAB, dtype=torch.uint8, device="cuda"),
           torch.full((cap, K // 32), 0xCD, dtype=torch.uint8, device="cuda"))
    st, ex, nt, q, s = mr.moe_sort_quant(idd, xd, N, B, quant, out=out, sorted_rows=True)
    st_t, ex_t, nt_t, _, _ = mr.moe_sort_quant(idd, xd, N, B, quant)
    for a, b in ((st, st_t), (ex, ex_t), (nt, nt_t)):
        assert np.array_equal(host(a), host(b))
    check_sort(ids, N, B, host(st), host(ex), host(nt))
    n = int(host(nt)[0])
    wq, ws = oracle.sorted_quant(x, k, host(st), n, quant)
    qh, sh = host(q), host(s)
    assert np.array_equal(qh[:n], wq), f"rows differ: {np.flatnonzero(np.any(qh[:n] != wq, 1))[:8]}"
    assert np.array_equal(sh[:n], ws)
    assert np.all(qh[n:] == 0xAB) and np.all(sh[n:] == 0xCD)
