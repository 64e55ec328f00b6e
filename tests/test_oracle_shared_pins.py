"""Pins of the oracle's shared-expert gate/up projection and SwiGLU
(oracle_shared_gate_up) and of its two helpers, the E4M3 decoder and the
rounding of a double to bf16.  Nothing here reuses the oracle's own
formulas: exact rationals, mpmath and the (separately pinned) E4M3 encoder
stand against it."""

from fractions import Fraction

import mpmath
import numpy as np
import pytest

import oracle
from decode_expert_routing_gb300 import inputs


def test_e4m3_decode_round_trips_through_the_encoder():
    """Every finite E4M3 code decodes to a value the (exhaustively pinned)
    encoder maps back to the same code; positive codes increase with their
    value; fixed points of the format hold; the NaN codes decode to NaN."""
    vals = []
    for c in range(256):
        v = oracle.e4m3_decode(c)
        if (c & 0x7F) == 0x7F:
            assert np.isnan(v)
            continue
        assert oracle.e4m3_encode(v) == c, hex(c)
        if c < 0x80:
            vals.append(v)
    assert all(a < b for a, b in zip(vals, vals[1:]))
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9 and oracle.e4m3_decode(0x08) == 2.0 ** -6
    assert oracle.e4m3_decode(0x78) == 256.0 and oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0xB8) == -1.0 and oracle.e4m3_decode(0xB0) == -0.5 and str(oracle.e4m3_decode(0x80)) == "-0.0"


def _bf16_nearest_exact(v):
    """bf16 bits nearest to v by exact comparison with both neighbours."""
    f = np.float32(v)
    u = int(np.array([f]).view(np.uint32)[0])
    lo = u & 0xFFFF0000
    cands = {lo, lo + 0x10000, lo - 0x10000}
    best = None
    for c in cands:
        if c < 0 or (c & 0x7F800000) == 0x7F800000:
            continue
        cv = Fraction(float(np.array([c], np.uint32).view(np.float32)[0]))
        d = abs(cv - Fraction(v))
        key = (d, (c >> 16) & 1)
        if best is None or key < best[0]:
            best = (key, c >> 16)
    return best[1]


def test_bf16_from_double_is_nearest_even():
    rng = np.random.default_rng(3)
    vals = list(rng.standard_normal(400) * 10.0 ** rng.integers(-40, 38, 400))
    vals += [1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -134,
             1.0 + 2.0 ** -8 + 2.0 ** -40, 0.0, -0.0]
    for v in vals:
        assert oracle.bf16_from_double(v) == _bf16_nearest_exact(v), v
    assert oracle.bf16_from_double(1 + 2.0 ** -8) == 0x3F80          # tie to the even code
    assert oracle.bf16_from_double(1 + 3 * 2.0 ** -8) == 0x3F82
    assert oracle.bf16_from_double(2.0 ** -134) == 0x0000            # tie with the smallest subnormal
    assert oracle.bf16_from_double(-0.0) == 0x8000


def _exact_h(x, codes, scale):
    """h as exact rationals: bf16 values times E4M3 values times 2^X."""
    M, K = x.shape
    R = codes.shape[0]
    xv = inputs.bf16_bits_to_f32(x).astype(np.float64)
    out = [[Fraction(0)] * R for _ in range(M)]
    for r in range(R):
        w = [Fraction(oracle.e4m3_decode(codes[r, k])) * Fraction(2) ** (int(scale[r, k // 32]) - 127)
             for k in range(K)]
        for m in range(M):
            out[m][r] = sum((Fraction(float(xv[m, k])) * w[k] for k in range(K)), Fraction(0))
    return out


def _act_bits(g, u):
    with mpmath.workdps(60):
        g, u = mpmath.mpf(g.numerator) / g.denominator, mpmath.mpf(u.numerator) / u.denominator
        a = g / (1 + mpmath.exp(-g)) * u
        return _bf16_nearest_exact(Fraction(str(mpmath.nstr(a, 50))))


@pytest.mark.parametrize("M,K,I", [(1, 32, 2), (3, 96, 4), (2, 64, 8)])
def test_shared_gate_up_against_exact_rationals(M, K, I):
    x, _ = inputs.router_inputs(M, K, 8, 7)
    codes, scale = inputs.shared_expert_weights(I, K)
    act, h = oracle.shared_gate_up(x, codes, scale)
    ex = _exact_h(x, codes, scale)
    for m in range(M):
        for r in range(2 * I):
            assert abs(Fraction(h[m, r]) - ex[m][r]) <= abs(ex[m][r]) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 200)
        for i in range(I):
            assert act[m, i] == _act_bits(ex[m][i], ex[m][I + i]), (m, i)


def test_shared_gate_up_closed_forms():
    """One-hot rows of x pick a column of W exactly; act is then silu of the
    gate weight times the up weight (a swapped gate/up would give silu(up) *
    gate); a zero gate row gives zero; scale bytes shift by exact powers of two."""
    I, K = 4, 64
    codes, scale = inputs.shared_expert_weights(I, K)
    x = np.zeros((K, K), np.uint16)
    for j in range(K):
        x[j, j] = 0x3F80  # 1.0
    act, h = oracle.shared_gate_up(x, codes, scale)
    for j in range(0, K, 7):
        for r in range(2 * I):
            w = oracle.e4m3_decode(codes[r, j]) * 2.0 ** (int(scale[r, j // 32]) - 127)
            assert h[j, r] == w
        for i in range(I):
            assert act[j, i] == _act_bits(Fraction(h[j, i]), Fraction(h[j, I + i]))
    c0 = codes.copy()
    c0[1] = 0  # gate row 1 all zero
    a0, _ = oracle.shared_gate_up(x[:3], c0, scale)
    assert np.all(a0[:, 1] & 0x7FFF == 0)
    s1 = scale.copy()
    s1[:I] += 1  # gate weights doubled: h of the gate rows doubles exactly
    _, h1 = oracle.shared_gate_up(x[:5], codes, s1)
    assert np.array_equal(h1[:, :I], 2 * h[:5, :I]) and np.array_equal(h1[:, I:], h[:5, I:])
