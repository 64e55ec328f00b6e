"""Pins of the oracle's router input on the norm's scale (CPU only).

The router takes the un-normalised residual rows, each token's rstd and the
norm weight, and forms xn = bf16((x * rstd) * s) with s = g (RMSNorm) or
1 + g (Gemma RMSNorm), both products in fp32.  These tests pin
oracle.norm_apply to facts that do not depend on its code: identities,
exact power-of-two scaling, hand-built rounding ties, a brute-force nearest
search over every finite bf16 code, an error bound, and the relation
between the two norm kinds.
"""

import numpy as np
import pytest

import oracle
from decode_expert_routing_gb300 import inputs


def bf16_val(bits):
    return inputs.bf16_bits_to_f32(np.asarray(bits, dtype=np.uint16)).astype(np.float64)


def all_finite_bf16():
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    return b[(b & 0x7F80) != 0x7F80]


def test_norm_identity_over_all_bf16():
    x = all_finite_bf16()
    K = x.shape[0]
    one = np.full(K, 0x3F80, dtype=np.uint16)    # 1.0
    zero = np.zeros(K, dtype=np.uint16)
    r = np.ones(1, dtype=np.float32)
    assert np.array_equal(oracle.norm_apply(x[None, :], r, one, "rms")[0], x)
    assert np.array_equal(oracle.norm_apply(x[None, :], r, zero, "gemma")[0], x)


@pytest.mark.parametrize("a,b", [(0, 0), (1, 0), (-3, 2), (2, -1), (5, 1), (-7, -2)])
def test_norm_powers_of_two_are_exact(a, b):
    x = inputs.normal_bf16((4, 256), 1.0, 6, 91)
    r = np.full(4, 2.0 ** a, dtype=np.float32)
    want = inputs.f64_to_bf16_bits(bf16_val(x) * 2.0 ** (a + b))   # exact scaling, no rounding
    g_rms = np.full(256, inputs.f64_to_bf16_bits(np.array([2.0 ** b]))[0], dtype=np.uint16)
    assert np.array_equal(oracle.norm_apply(x, r, g_rms, "rms"), want)
    g_gem = inputs.f64_to_bf16_bits(np.full(256, 2.0 ** b - 1.0))   # 1 + g = 2^b, exact in bf16
    assert np.array_equal(oracle.norm_apply(x, r, g_gem, "gemma"), want)


# (x, rstd, expected bf16 bits) with s = 1: ties go to the even code
TIES = [
    (1.0, 1 + 2 ** -8, 0x3F80),                    # halfway between 1 and 1 + 2^-7: even is 1
    (1.0, 1 + 3 * 2 ** -8, 0x3F82),                # halfway between 1 + 2^-7 and 1 + 2^-6: even is 0x3F82
    (-1.0, 1 + 2 ** -8, 0xBF80),
    (-1.0, 1 + 3 * 2 ** -8, 0xBF82),
    (1.0, 1 + 2 ** -8 + 2 ** -20, 0x3F81),         # just past the midpoint: up
    (1.0, 1 + 2 ** -8 - 2 ** -20, 0x3F80),         # just short of it: down
    (1 + 2 ** -7, 1 + 2 ** -8, 0x3F82),            # 1 + 3 * 2^-8 + 2^-15: past the midpoint
]


@pytest.mark.parametrize("xv,rv,want", TIES)
def test_norm_ties_round_to_even(xv, rv, want):
    x = inputs.f64_to_bf16_bits(np.array([[xv]]))
    assert bf16_val(x)[0, 0] == xv
    r = np.array([rv], dtype=np.float32)
    assert float(r[0]) == rv                       # the rstd is exact in fp32
    got = oracle.norm_apply(x, r, np.array([0x3F80], dtype=np.uint16), "rms")
    assert int(got[0, 0]) == want


def test_norm_subnormal_results_round_to_nearest():
    # x * rstd lands among bf16 subnormals (quantum 2^-133): 3 * 2^-134 is a
    # tie between 2^-133 (odd code 1) and 2^-132 (even code 2) -> 2;
    # 2^-134 is a tie between 0 and 2^-133 -> 0; 5 * 2^-135 -> 2^-133 * 1.25 -> code 1
    cases = [(3.0, 2.0 ** -134, 0x0002), (1.0, 2.0 ** -134, 0x0000), (5.0, 2.0 ** -135, 0x0001),
             (-3.0, 2.0 ** -134, 0x8002)]
    for xv, rv, want in cases:
        x = inputs.f64_to_bf16_bits(np.array([[xv]]))
        r = np.array([rv], dtype=np.float32)
        assert float(r[0]) == rv
        got = oracle.norm_apply(x, r, np.array([0x3F80], dtype=np.uint16), "rms")
        assert int(got[0, 0]) == want, (xv, rv, hex(int(got[0, 0])))


def _nearest_bf16_brute(p: np.ndarray) -> np.ndarray:
    """Nearest finite bf16 code to each float, ties to the even code, by a
    search over the sorted table of every finite bf16 value."""
    codes = all_finite_bf16()
    vals = bf16_val(codes)
    order = np.lexsort((codes, vals))
    vals, codes = vals[order], codes[order]
    out = np.empty(p.shape[0], dtype=np.uint16)
    for i, v in enumerate(p.astype(np.float64)):
        j = np.searchsorted(vals, v)
        cand = []
        for jj in (j - 2, j - 1, j, j + 1):
            if 0 <= jj < len(vals):
                cand.append((abs(vals[jj] - v), int(codes[jj]) & 1, int(codes[jj])))
        cand.sort()
        best = [c for c in cand if c[0] == cand[0][0]]
        if v == 0.0:
            out[i] = 0x8000 if np.signbit(v) else 0x0000
            continue
        # among equally near codes of the right sign, the even one
        best = [c for c in best if (c[2] >> 15) == (1 if v < 0 else 0)] or best
        best.sort(key=lambda c: c[1])
        out[i] = best[0][2]
    return out


def test_norm_rounding_matches_brute_force_nearest():
    rng = np.random.default_rng(7)
    M, K = 3, 400
    x = inputs.normal_bf16((M, K), 2.0, 6, 92)
    r = (rng.uniform(0.01, 4.0, M)).astype(np.float32)
    g = inputs.normal_bf16((K,), 0.1, 6, 93)
    for kind in ("rms", "gemma"):
        got = oracle.norm_apply(x, r, g, kind)
        s = bf16_val(g).astype(np.float32)
        if kind == "gemma":
            s = (np.float32(1.0) + s).astype(np.float32)
        t = (bf16_val(x).astype(np.float32) * r[:, None]).astype(np.float32)   # fp32 products, IEEE
        p = (t * s[None, :]).astype(np.float32)
        want = _nearest_bf16_brute(p.ravel()).reshape(M, K)
        assert np.array_equal(got, want), kind


def test_norm_error_bound_against_exact_product():
    x = inputs.normal_bf16((8, 512), 1.0, 6, 94)
    r = np.linspace(0.05, 3.0, 8).astype(np.float32)
    g = inputs.normal_bf16((512,), 0.1, 6, 95)
    got = bf16_val(oracle.norm_apply(x, r, g, "gemma"))
    exact = bf16_val(x) * r.astype(np.float64)[:, None] * (1.0 + bf16_val(g))[None, :]
    # bf16 keeps 8 significant bits (half an ulp: 2^-8 relative) plus two
    # fp32 roundings on the way (2^-24 each)
    assert np.all(np.abs(got - exact) <= (2.0 ** -8 + 2.0 ** -22) * np.abs(exact) + 1e-38)
    # and the result is one of the two bf16 neighbours of the exact value
    assert np.all(np.abs(got - exact) <= np.abs(exact) * 2.0 ** -7)


def test_norm_gemma_is_rms_of_one_plus_g_when_exact():
    x = inputs.normal_bf16((2, 128), 1.0, 6, 96)
    r = np.array([0.37, 1.9], dtype=np.float32)
    gv = np.array([0.0, 0.5, -0.5, 2.0 ** -7, -(2.0 ** -7), 0.25, 3.0, -0.75] * 16)
    g = inputs.f64_to_bf16_bits(gv)
    one_plus = inputs.f64_to_bf16_bits(1.0 + gv)   # exact: every 1 + g here is a bf16 value
    assert np.array_equal(bf16_val(one_plus), 1.0 + gv)
    assert np.array_equal(oracle.norm_apply(x, r, g, "gemma"), oracle.norm_apply(x, r, one_plus, "rms"))


def test_norm_inputs_recipe():
    s, r, g = inputs.norm_inputs(64, 6144)
    s2, r2, g2 = inputs.norm_inputs(64, 6144)
    assert np.array_equal(s, s2) and np.array_equal(r, r2) and np.array_equal(g, g2)
    assert r.dtype == np.float32 and np.all(r > 1.0 / 8.0 - 1e-6) and np.all(r < 2.0 + 1e-6)
    xn = bf16_val(oracle.norm_apply(s, r, g, "gemma"))
    rms = np.sqrt((xn ** 2).mean(axis=1))
    assert np.all(np.abs(rms - 1.0) < 0.05)        # the norm's output has unit scale per row
    assert abs(bf16_val(g).std() - 0.1) < 0.01


def test_norm_product_order_is_x_times_rstd_first():
    # (x * rstd) * s and x * (rstd * s) differ in fp32 now and then, and the
    # bf16 rounding shows it only near a bf16 midpoint: search seeded triples
    # for such cases and check the oracle takes the (x * rstd) * s order
    rng = np.random.default_rng(11)
    n = 1 << 20
    x = inputs.f64_to_bf16_bits(rng.standard_normal(n))
    xv = bf16_val(x).astype(np.float32)
    r = rng.uniform(0.05, 4.0, n).astype(np.float32)
    s = (np.float32(1.0) + bf16_val(inputs.f64_to_bf16_bits(rng.standard_normal(n) * 0.1)).astype(np.float32))
    p1 = ((xv * r).astype(np.float32) * s).astype(np.float32)
    p2 = (xv * (r * s).astype(np.float32)).astype(np.float32)
    diff = np.nonzero(p1 != p2)[0]
    hi1, hi2 = p1.view(np.uint32) >> 16, p2.view(np.uint32) >> 16
    lo1 = p1.view(np.uint32) & 0xFFFF
    near_mid = diff[(np.abs(lo1[diff].astype(np.int64) - 0x8000) <= 1) | (hi1[diff] != hi2[diff])]
    idx = near_mid[:64]
    want1 = _nearest_bf16_brute(p1[idx])
    want2 = _nearest_bf16_brute(p2[idx])
    assert np.any(want1 != want2)                  # the sample tells the two orders apart
    g = inputs.f64_to_bf16_bits(s[idx].astype(np.float64) - 1.0)
    assert np.array_equal(np.float32(1.0) + bf16_val(g).astype(np.float32), s[idx])
    for j, i in enumerate(idx):
        got = oracle.norm_apply(x[i:i + 1].reshape(1, 1), r[i:i + 1], g[j:j + 1], "gemma")
        assert int(got[0, 0]) == int(want1[j])
