"""Helpers shared by the GPU parity tests (not a test module)."""

import numpy as np

import oracle
from decode_expert_routing_gb300 import inputs

LOGIT_RTOL = 1e-4      # |gpu - ref| <= 1e-4 * (1 + |ref|)
WEIGHT_ATOL = 1e-6     # routing weights, absolute


def torch_mod():
    import torch
    return torch


def to_dev_bf16(u16):
    torch = torch_mod()
    t = torch.from_numpy(np.ascontiguousarray(u16).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def to_dev(a):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def assert_logits_close(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref) / (1.0 + np.abs(ref))
    assert err.max() <= LOGIT_RTOL, f"max rel err {err.max():.3e}"
    return err.max()


def check_gate(logits_host, ids, wts, topk, scoring, bias=None, renormalize=True):
    """Gate outputs against the oracle run on the same (GPU-produced) logits."""
    rid, rw = oracle.route_topk(logits_host, topk, scoring, bias, renormalize)
    ids, wts = np.asarray(ids), np.asarray(wts)
    assert np.array_equal(ids, rid), f"ids differ in {np.sum(np.any(ids != rid, 1))} rows"
    assert np.max(np.abs(wts.astype(np.float64) - rw)) <= WEIGHT_ATOL
    return rid, rw


def check_sort(ids, N, block, st, ex, nt):
    rst, rex, rnt = oracle.moe_sort(np.asarray(ids, np.int32), N, block)
    st, ex = np.asarray(st), np.asarray(ex)
    assert int(np.asarray(nt).reshape(-1)[0]) == rnt
    assert np.array_equal(st, rst), f"sorted_token_ids differ at {np.flatnonzero(st != rst)[:8]}"
    assert np.array_equal(ex, rex), f"expert_ids differ at {np.flatnonzero(ex != rex)[:8]}"


def check_quant(x_u16, q, s):
    rq, rs = oracle.mxfp8_quant(x_u16)
    q, s = np.asarray(q), np.asarray(s)
    assert np.array_equal(s, rs), f"scales differ at {np.argwhere(s != rs)[:8].tolist()}"
    assert np.array_equal(q, rq), f"codes differ at {np.argwhere(q != rq)[:8].tolist()}"
