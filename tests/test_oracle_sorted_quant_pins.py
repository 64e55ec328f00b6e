"""Pins of the oracle's stage-1 activations in sorted order
(oracle_sorted_quant): a worked example by hand, and properties on random
routings that tie each output row to the token-order quantisation."""

import os

import numpy as np
import pytest

import oracle
from decode_expert_routing_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    out = {}
    for line in open(os.path.join(GOLDEN, "sorted_quant_example.txt")):
        if line.strip() and not line.startswith("#"):
            key, *vals = line.split()
            out[key] = [int(v) for v in vals]
    return out


def test_sorted_quant_worked_example():
    g = _golden()
    x = np.zeros((2, 32), np.uint16)
    x[0], x[1] = 0x3F80, 0xC000
    ids = np.array([[2, 0], [0, 1]], np.int32)
    st, ex, nt = oracle.moe_sort(ids, 3, 2)
    assert st.tolist() == g["sorted_token_ids"] and nt == g["num_tokens_post_padded"][0]
    q, s = oracle.sorted_quant(x, 2, st, nt, "mxfp8")
    assert q.shape == (6, 32) and np.all(q == q[:, :1])  # constant rows
    assert q[:, 0].tolist() == g["mxfp8_code"] and s[:, 0].tolist() == g["mxfp8_scale"]
    q4, s4 = oracle.sorted_quant(x, 2, st, nt, "mxfp4")
    assert q4.shape == (6, 16) and np.all(q4 == q4[:, :1])
    assert q4[:, 0].tolist() == g["mxfp4_byte"] and s4[:, 0].tolist() == g["mxfp4_scale"]


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("M,k,N,B", [(1, 8, 128, 16), (16, 8, 128, 16), (64, 8, 128, 64), (7, 3, 9, 4)])
def test_sorted_quant_rows_are_token_rows(fmt, M, k, N, B):
    """Row p equals the token-order quantisation of token sorted[p] // k;
    padding rows are zero; every real assignment's token appears once per
    assignment; the row count is num_tokens_post_padded."""
    K = 256
    x = inputs.prefill_x(M, K)
    rng = np.random.default_rng(M * 31 + k)
    ids = np.stack([rng.choice(N, k, replace=False) for _ in range(M)]).astype(np.int32)
    st, _, nt = oracle.moe_sort(ids, N, B)
    q, s = oracle.sorted_quant(x, k, st, nt, fmt)
    tq, ts = (oracle.mxfp8_quant if fmt == "mxfp8" else oracle.mxfp4_quant)(x)
    assert q.shape[0] == nt == s.shape[0]
    seen = np.zeros(M, int)
    for p in range(nt):
        f = int(st[p])
        if f < M * k:
            assert np.array_equal(q[p], tq[f // k]) and np.array_equal(s[p], ts[f // k])
            seen[f // k] += 1
        else:
            assert not q[p].any() and not s[p].any()
    assert np.all(seen == k)
