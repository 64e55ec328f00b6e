"""CPU oracle for the MoE decode routing path (ctypes wrapper over oracle.c).

TEST INFRASTRUCTURE ONLY.  The tests, the package smoke check and the
benchmark's CPU-baseline leg are the only callers; the CUDA library never
imports, links or runs anything here, and this module never imports the CUDA
library.  ``build()`` compiles oracle.c with gcc (no CUDA needed).

All arrays are numpy: bf16 tensors travel as uint16 bit patterns.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain C11, no fp contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                        "-fno-fast-math", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int, ctypes.c_int64
        lib.oracle_router_gemv.argtypes = [P, i64, P, P, i32, i32, i32]
        lib.oracle_topk_softmax.argtypes = [P, i32, i32, i32, i32, P, P]
        lib.oracle_topk_sigmoid.argtypes = [P, P, i32, i32, i32, i32, P, P]
        lib.oracle_sigmoid_f32.argtypes = [ctypes.c_float]
        lib.oracle_sigmoid_f32.restype = ctypes.c_float
        lib.oracle_sigmoid_f32_array.argtypes = [P, i64, P]
        lib.oracle_sort_capacity.argtypes = [i32, i32, i32, i32]
        lib.oracle_sort_capacity.restype = i64
        lib.oracle_moe_sort.argtypes = [P, i32, i32, i32, i32, P, P, P, i64]
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode_array.argtypes = [P, i64, P]
        lib.oracle_mxfp8_quant.argtypes = [P, i64, i32, i32, P, P]
        lib.oracle_bf16_round.argtypes = [ctypes.c_float]
        lib.oracle_bf16_round.restype = ctypes.c_uint16
        lib.oracle_norm_apply.argtypes = [P, i64, P, P, i32, i32, i32, P]
        lib.oracle_e2m1_encode.argtypes = [ctypes.c_double]
        lib.oracle_e2m1_encode.restype = ctypes.c_uint8
        lib.oracle_e2m1_encode_array.argtypes = [P, i64, P]
        lib.oracle_mxfp4_quant.argtypes = [P, i64, i32, i32, P, P]
        lib.oracle_sorted_quant.argtypes = [P, i64, i32, i32, i32, P, i32, i32, P, P]
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
        lib.oracle_bf16_from_double.restype = ctypes.c_uint16
        lib.oracle_shared_gate_up.argtypes = [P, i64, P, P, i32, i32, i32, P, P]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a, dtype=dtype))


def router_gemv(x_bf16: np.ndarray, w_bf16: np.ndarray) -> np.ndarray:
    """fp32 logits [M, N] of x [M, K] (bf16 bits) times W [N, K] (bf16 bits)."""
    x = _c(x_bf16, np.uint16)
    w = _c(w_bf16, np.uint16)
    M, K = x.shape
    N, K2 = w.shape
    assert K == K2
    out = np.empty((M, N), dtype=np.float32)
    _load().oracle_router_gemv(_ptr(x), K, _ptr(w), _ptr(out), M, N, K)
    return out


def route_topk(logits: np.ndarray, topk: int, scoring: str = "softmax", bias=None,
               renormalize: bool = True):
    """(topk_ids int32 [M, k], topk_weights float32 [M, k])."""
    lg = _c(logits, np.float32)
    M, N = lg.shape
    ids = np.empty((M, topk), dtype=np.int32)
    wts = np.empty((M, topk), dtype=np.float32)
    lib = _load()
    if scoring == "softmax":
        lib.oracle_topk_softmax(_ptr(lg), M, N, topk, int(renormalize), _ptr(ids), _ptr(wts))
    elif scoring == "sigmoid":
        b = None if bias is None else _c(bias, np.float32)
        lib.oracle_topk_sigmoid(_ptr(lg), None if b is None else _ptr(b), M, N, topk,
                                int(renormalize), _ptr(ids), _ptr(wts))
    else:
        raise ValueError(scoring)
    return ids, wts


def sigmoid_f32(values) -> np.ndarray:
    """The correctly rounded fp32 sigmoid 1 / (1 + e^-l), element by element."""
    v = _c(values, np.float32).ravel()
    out = np.empty(v.shape[0], dtype=np.float32)
    _load().oracle_sigmoid_f32_array(_ptr(v), v.shape[0], _ptr(out))
    return out.reshape(np.shape(values))


def sort_capacity(M: int, topk: int, N: int, block: int) -> int:
    return int(_load().oracle_sort_capacity(M, topk, N, block))


def moe_sort(topk_ids: np.ndarray, N: int, block: int):
    """(sorted_token_ids, expert_ids, num_tokens_post_padded) for ids [M, k]."""
    ids = _c(topk_ids, np.int32)
    M, k = ids.shape
    cap = sort_capacity(M, k, N, block)
    st = np.empty(cap, dtype=np.int32)
    ex = np.empty(cap // block, dtype=np.int32)
    nt = np.empty(1, dtype=np.int32)
    _load().oracle_moe_sort(_ptr(ids), M, k, N, block, _ptr(st), _ptr(ex), _ptr(nt), cap)
    return st, ex, int(nt[0])


def e4m3_encode(v: float) -> int:
    return int(_load().oracle_e4m3_encode(float(v)))


def e4m3_encode_array(values) -> np.ndarray:
    v = _c(values, np.float64).ravel()
    out = np.empty(v.shape[0], dtype=np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(v), v.shape[0], _ptr(out))
    return out.reshape(np.shape(values))


def mxfp8_quant(x_bf16: np.ndarray):
    """(q uint8 [M, K] e4m3 codes, scale uint8 [M, K/32] e8m0 bytes)."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    assert K % 32 == 0
    q = np.empty((M, K), dtype=np.uint8)
    s = np.empty((M, K // 32), dtype=np.uint8)
    _load().oracle_mxfp8_quant(_ptr(x), K, M, K, _ptr(q), _ptr(s))
    return q, s


def route_sort_quant(x_bf16, w_bf16, topk, block, scoring="softmax", bias=None,
                     renormalize=True):
    """The whole path composed from the steps above (dict of outputs)."""
    logits = router_gemv(x_bf16, w_bf16)
    ids, wts = route_topk(logits, topk, scoring, bias, renormalize)
    st, ex, nt = moe_sort(ids, w_bf16.shape[0], block)
    q, s = mxfp8_quant(x_bf16)
    return dict(logits=logits, topk_ids=ids, topk_weights=wts, sorted_token_ids=st,
                expert_ids=ex, num_tokens_post_padded=nt, q=q, scale=s)


NORM_KINDS = {"rms": 0, "gemma": 1}


def bf16_round(f: float) -> int:
    """bf16 bits of the nearest bf16 to the float32 value f (ties to even)."""
    return int(_load().oracle_bf16_round(float(np.float32(f))))


def norm_apply(x_bf16: np.ndarray, rstd: np.ndarray, g_bf16: np.ndarray, kind: str = "gemma") -> np.ndarray:
    """xn = bf16((x * rstd[m]) * s[k]) in fp32 steps, s = g or 1 + g (bf16 bits [M, K])."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    r = _c(rstd, np.float32).ravel()
    g = _c(g_bf16, np.uint16).ravel()
    assert r.shape[0] == M and g.shape[0] == K
    out = np.empty((M, K), dtype=np.uint16)
    _load().oracle_norm_apply(_ptr(x), K, _ptr(r), _ptr(g), NORM_KINDS[kind], M, K, _ptr(out))
    return out


def route_sort_quant_norm(sres_bf16, rstd, g_bf16, kind, w_bf16, topk, block, scoring="softmax",
                          bias=None, renormalize=True):
    """The route of norm_apply's output (dict of outputs plus "xn")."""
    xn = norm_apply(sres_bf16, rstd, g_bf16, kind)
    out = route_sort_quant(xn, w_bf16, topk, block, scoring, bias, renormalize)
    out["xn"] = xn
    return out


def e2m1_encode(v: float) -> int:
    return int(_load().oracle_e2m1_encode(float(v)))


def e2m1_encode_array(values) -> np.ndarray:
    v = _c(values, np.float64).ravel()
    out = np.empty(v.shape[0], dtype=np.uint8)
    _load().oracle_e2m1_encode_array(_ptr(v), v.shape[0], _ptr(out))
    return out.reshape(np.shape(values))


def mxfp4_quant(x_bf16: np.ndarray):
    """(q uint8 [M, K/2] packed e2m1 codes, scale uint8 [M, K/32] e8m0 bytes)."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    assert K % 32 == 0
    q = np.empty((M, K // 2), dtype=np.uint8)
    s = np.empty((M, K // 32), dtype=np.uint8)
    _load().oracle_mxfp4_quant(_ptr(x), K, M, K, _ptr(q), _ptr(s))
    return q, s


def sorted_quant(x_bf16: np.ndarray, topk: int, sorted_token_ids: np.ndarray, num_tokens_post_padded: int,
                 fmt: str = "mxfp8"):
    """Stage-1 activations in sorted order: (q uint8 [ntpp, K] or [ntpp, K/2],
    scale uint8 [ntpp, K/32]); row p quantises x[sorted_token_ids[p] // topk],
    padding rows are zero."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    st = _c(sorted_token_ids, np.int32)
    n = int(num_tokens_post_padded)
    fp4 = {"mxfp8": 0, "mxfp4": 1}[fmt]
    q = np.empty((n, K // 2 if fp4 else K), dtype=np.uint8)
    s = np.empty((n, K // 32), dtype=np.uint8)
    _load().oracle_sorted_quant(_ptr(x), K, M, K, topk, _ptr(st), n, fp4, _ptr(q), _ptr(s))
    return q, s


def e4m3_decode(code: int) -> float:
    """Exact value of an E4M3 code (NaN for S.1111.111)."""
    return float(_load().oracle_e4m3_decode(int(code)))


def bf16_from_double(v: float) -> int:
    """bf16 bits of the bf16 value nearest to the double v (ties to even)."""
    return int(_load().oracle_bf16_from_double(float(v)))


def shared_gate_up(x_bf16: np.ndarray, w13_codes: np.ndarray, w13_scale: np.ndarray):
    """The shared expert's gate/up projection and SwiGLU: (act bf16 bits
    [M, I], h float64 [M, 2I]) for x [M, K] (bf16 bits), w13 E4M3 codes
    [2I, K] (gate rows first) and E8M0 scale bytes [2I, K/32]."""
    x = _c(x_bf16, np.uint16)
    w = _c(w13_codes, np.uint8)
    sc = _c(w13_scale, np.uint8)
    M, K = x.shape
    R, K2 = w.shape
    assert K == K2 and R % 2 == 0 and sc.shape == (R, K // 32)
    act = np.empty((M, R // 2), dtype=np.uint16)
    h = np.empty((M, R), dtype=np.float64)
    _load().oracle_shared_gate_up(_ptr(x), K, _ptr(w), _ptr(sc), M, K, R // 2, _ptr(act), _ptr(h))
    return act, h
