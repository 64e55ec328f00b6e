"""Pins of the oracle's MXFP4 quantiser (CPU only): the E2M1 encoder against
an independent per-binade round-to-nearest-even over every bf16 pattern at
several scales, every E2M1 value round-tripping, monotonicity and the
half-spacing error bound, and hand-derived blocks (tests/golden)."""

import os

import numpy as np
import pytest

import oracle
from decode_expert_routing_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def bf16_val(bits):
    return inputs.bf16_bits_to_f32(np.asarray(bits, dtype=np.uint16)).astype(np.float64)


def e2m1_by_binade(v: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even per binade, written independently of the
    oracle's nearest-of-eight search: quantum 0.5 below 2, 1 in [2, 4),
    2 in [4, 6]; codes count quanta from the binade's start; saturate at 6."""
    a = np.abs(v)
    code = np.empty(a.shape, dtype=np.int64)
    lo = a < 2.0
    code[lo] = np.rint(a[lo] / 0.5).astype(np.int64)                  # 0..4 (4 = 2.0)
    mid = (a >= 2.0) & (a < 4.0)
    code[mid] = np.rint(a[mid]).astype(np.int64) + 2                  # 2 -> 4, 3 -> 5, 4 -> 6
    hi = (a >= 4.0) & (a <= 6.0)
    code[hi] = np.rint(a[hi] / 2.0).astype(np.int64) + 4              # 4 -> 6, 6 -> 7
    code[a > 6.0] = 7
    return (code | (np.signbit(v).astype(np.int64) << 3)).astype(np.uint8)


def test_e2m1_values_round_trip():
    for c, m in enumerate(E2M1):
        assert oracle.e2m1_encode(m) == c
        assert oracle.e2m1_encode(-m) == c | 8


@pytest.mark.parametrize("scale_exp", [-130, -20, -8, -3, 0, 2, 7, 30, 120])
def test_e2m1_encoder_exhaustive_over_bf16_patterns(scale_exp):
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    b = b[(b & 0x7F80) != 0x7F80]                                     # finite
    v = bf16_val(b) * 2.0 ** scale_exp                                 # exact in float64
    got = oracle.e2m1_encode_array(v)
    assert np.array_equal(got, e2m1_by_binade(v))


def test_e2m1_monotone_and_error_bound():
    v = np.linspace(-8.0, 8.0, 20001)
    codes = oracle.e2m1_encode_array(v)
    val = np.array([(-1.0 if c & 8 else 1.0) * E2M1[c & 7] for c in codes])
    assert np.all(np.diff(val) >= 0)
    inside = np.abs(v) <= 6.0
    spacing = np.where(np.abs(v) < 2.0, 0.5, np.where(np.abs(v) < 4.0, 1.0, 2.0))
    assert np.all(np.abs(val - v)[inside] <= spacing[inside] / 2 + 1e-12)
    assert np.all(np.abs(val[~inside]) == 6.0)


def _golden_blocks(name):
    cases, cur = {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] == "case":
                cur = parts[1]
                cases[cur] = {"elems": [], "scale": None}
            elif parts[0] == "scale":
                cases[cur]["scale"] = int(parts[1], 16)
            else:
                cases[cur]["elems"].append((int(parts[0]), float(parts[1]), int(parts[2], 16)))
    return cases


GOLD = _golden_blocks("mxfp4_blocks.txt")


@pytest.mark.parametrize("case", sorted(GOLD))
def test_mxfp4_golden_blocks(case):
    g = GOLD[case]
    vals = np.zeros(32)
    codes = np.zeros(32, dtype=np.uint8)
    for i, v, c in g["elems"]:
        vals[i] = v
        codes[i] = c
    x = inputs.f64_to_bf16_bits(vals)
    for i, v, _ in g["elems"]:
        assert bf16_val(x[i]) == v or (v == 0.0 and np.signbit(v)), (case, i)
    q, s = oracle.mxfp4_quant(x[None, :])
    assert int(s[0, 0]) == g["scale"]
    want = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
    assert q[0].tolist() == want.tolist(), case


def test_mxfp4_scale_rule_and_packing_on_random_rows():
    x = inputs.prefill_x(4, 256)
    q, s = oracle.mxfp4_quant(x)
    xv = bf16_val(x).reshape(4, 8, 32)
    amax = np.abs(xv).max(axis=2)
    X = np.floor(np.log2(amax)).astype(int) - 2
    assert np.array_equal(s.astype(int) - 127, X)
    # every block's largest element scales into [4, 8): code 6 or 7
    lo = q & 0xF
    hi = q >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(4, 8, 32)
    imax = np.abs(xv).argmax(axis=2)
    top = np.take_along_axis(codes, imax[..., None], axis=2)[..., 0] & 7
    assert np.all((top == 6) | (top == 7))
    # dequantised values sit within half a quantum (or saturate)
    deq = np.array([E2M1[c & 7] for c in codes.ravel()]).reshape(codes.shape)
    deq = np.where(codes & 8, -deq, deq) * (2.0 ** X)[..., None]
    scaled = np.abs(xv) / (2.0 ** X)[..., None]
    quantum = np.where(scaled < 2, 0.5, np.where(scaled < 4, 1.0, 2.0)) * (2.0 ** X)[..., None]
    ok = (np.abs(deq - xv) <= quantum / 2 + 1e-30) | (scaled > 6.0)
    assert np.all(ok)
