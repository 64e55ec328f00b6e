"""Pins of the CPU oracle to things other than itself (CPU only).

Each test checks an oracle function against what the mathematics or a
hand-worked example fixes: exact integer sums, one-hot operands, closed forms,
brute force over every candidate on tiny inputs, invariants, an independent
library conversion, and the hand-derived fixtures in tests/golden/.  The set
is chosen so that a dropped term, a wrong sign, a swapped index or a
transposed operand in the oracle fails at least one of them.
"""

import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from decode_expert_routing_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(vals):
    return inputs.f64_to_bf16_bits(np.asarray(vals, dtype=np.float64))


def bf16_val(bits):
    return inputs.bf16_bits_to_f32(bits).astype(np.float64)


# ---------------------------------------------------------------- GEMV


def test_gemv_exact_small_integers():
    """Integer-valued operands: every partial sum is exact, so the fp32 logit
    must equal the exact integer dot product."""
    rng = np.random.default_rng(1)
    M, N, K = 3, 5, 64
    xv = rng.integers(-8, 9, size=(M, K)).astype(np.float64)
    wv = rng.integers(-8, 9, size=(N, K)).astype(np.float64)
    got = oracle.router_gemv(bf16(xv), bf16(wv))
    for m in range(M):
        for n in range(N):
            exact = sum(int(xv[m, k]) * int(wv[n, k]) for k in range(K))
            assert got[m, n] == np.float32(exact)


def _round_fraction_to_f32(fr: Fraction) -> np.float32:
    """Correctly rounded float32 of an exact rational (nearest, ties to even)."""
    if fr == 0:
        return np.float32(0.0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)
    q = a / (Fraction(2) ** (e - 23))
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return np.float32(sign * math.ldexp(n, e - 23))


def test_gemv_correctly_rounded_against_exact_rationals():
    """General bf16 operands: the exact dot product (as a rational) rounded
    once to fp32 must match the oracle (fp64 accumulation error is ~1e-16
    relative, far below half an fp32 ulp except on astronomically rare
    midpoints)."""
    x = inputs.normal_bf16((2, 96), 1.0, 99, 1)
    w = inputs.normal_bf16((7, 96), 0.02, 99, 2)
    got = oracle.router_gemv(x, w)
    xf, wf = bf16_val(x), bf16_val(w)
    for m in range(2):
        for n in range(7):
            exact = sum(Fraction(float(xf[m, k])) * Fraction(float(wf[n, k])) for k in range(96))
            assert got[m, n] == _round_fraction_to_f32(exact)


def test_gemv_one_hot_rows_pick_columns():
    """W row n = e_{j(n)} gives logits[m, n] = x[m, j(n)] exactly; with
    M != N != K this also catches a transposed operand or swapped index."""
    M, N, K = 4, 6, 40
    x = inputs.normal_bf16((M, K), 1.0, 98, 1)
    cols = [3, 0, 39, 17, 17, 8]
    w = np.zeros((N, K), dtype=np.uint16)
    for n, j in enumerate(cols):
        w[n, j] = 0x3F80  # bf16 1.0
    got = oracle.router_gemv(x, w)
    want = bf16_val(x)[:, cols].astype(np.float32)
    assert np.array_equal(got, want)


def test_gemv_powers_of_two_exact_and_sign():
    """Powers of two of mixed sign: exact sums, sign errors show."""
    K = 32
    x = np.array([[(-1) ** k * 2.0 ** (k % 5) for k in range(K)]])
    w = np.array([[2.0 ** -(k % 3) for k in range(K)], [-(2.0 ** (k % 4)) for k in range(K)]])
    got = oracle.router_gemv(bf16(x), bf16(w))
    want = x @ w.T  # exact: all terms are small dyadic rationals
    assert np.array_equal(got, want.astype(np.float32))


def test_gemv_identical_rows_identical_logits():
    x, w = inputs.router_inputs(3, 256, 64, 97)
    w = inputs.tied_gate(w, ((10, 11), (50, 51)))
    got = oracle.router_gemv(x, w)
    assert np.array_equal(got[:, 10].view(np.uint32), got[:, 11].view(np.uint32))
    assert np.array_equal(got[:, 50].view(np.uint32), got[:, 51].view(np.uint32))


# ---------------------------------------------------------------- top-k


def _selection_is_valid(key, sel):
    """Every selected key beats every unselected one; equal keys at the
    boundary go to the lower id."""
    sel = set(sel)
    for s in sel:
        for u in range(len(key)):
            if u in sel:
                continue
            if not (key[s] > key[u] or (key[s] == key[u] and s < u)):
                return False
    return True


@pytest.mark.parametrize("seed", range(12))
def test_topk_brute_force_over_all_subsets(seed):
    """For N <= 10, k <= 4 (with forced ties): exactly one subset satisfies
    the selection invariant, and it is the oracle's."""
    rng = np.random.default_rng(seed)
    N = int(rng.integers(4, 11))
    k = int(rng.integers(1, min(4, N) + 1))
    logits = rng.integers(-3, 4, size=(1, N)).astype(np.float32) * np.float32(0.5)
    ids, _ = oracle.route_topk(logits, k)
    valid = [c for c in itertools.combinations(range(N), k) if _selection_is_valid(logits[0], c)]
    assert len(valid) == 1
    assert set(ids[0].tolist()) == set(valid[0])
    keys = logits[0][ids[0]]
    for a in range(k - 1):  # slot order: key descending, then id ascending
        assert keys[a] > keys[a + 1] or (keys[a] == keys[a + 1] and ids[0][a] < ids[0][a + 1])


def test_topk_softmax_weights_sum_and_closed_form():
    rng = np.random.default_rng(5)
    lg = rng.standard_normal((16, 128)).astype(np.float32) * 1.5
    ids, w = oracle.route_topk(lg, 8)
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) <= 8 * 2.0 ** -24)
    for m in range(16):
        sel = lg[m, ids[m]].astype(np.float64)
        ref = np.exp(sel - sel.max()) / np.exp(sel - sel.max()).sum()
        assert np.max(np.abs(w[m] - ref)) <= 1e-7
    # not renormalised: the weights are the full softmax probabilities
    ids2, w2 = oracle.route_topk(lg, 128, renormalize=False)
    full = np.exp(lg.astype(np.float64) - lg.max(1, keepdims=True))
    full /= full.sum(1, keepdims=True)
    for m in range(16):
        assert np.max(np.abs(w2[m] - full[m, ids2[m]])) <= 1e-7


def test_topk_all_equal_logits():
    lg = np.full((3, 32), 0.25, dtype=np.float32)
    ids, w = oracle.route_topk(lg, 8)
    assert np.array_equal(ids, np.tile(np.arange(8, dtype=np.int32), (3, 1)))
    assert np.all(w == np.float32(1.0 / 8))


def test_topk_signed_zero_is_a_tie():
    lg = np.array([[-0.0, 0.0, -1.0, -0.0]], dtype=np.float32)
    ids, _ = oracle.route_topk(lg, 2)
    assert ids[0].tolist() == [0, 1]


def _golden_kv(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                key, *vals = line.split()
                out[key] = vals
    return out


def test_topk_golden_examples():
    g = _golden_kv("topk_examples.txt")
    lg = np.array([[float(v) for v in g["softmax_logits"]]], dtype=np.float32)
    ids, w = oracle.route_topk(lg, int(g["softmax_k"][0]))
    assert ids[0].tolist() == [int(v) for v in g["softmax_ids"]]
    want = [eval(expr, {"exp": math.exp}) for expr in g["softmax_weights"]]
    assert np.max(np.abs(w[0] - np.array(want))) <= 1e-7
    lg = np.array([[float(v) for v in g["sigmoid_logits"]]], dtype=np.float32)
    bias = np.array([float(v) for v in g["sigmoid_bias"]], dtype=np.float32)
    ids, w = oracle.route_topk(lg, int(g["sigmoid_k"][0]), "sigmoid", bias)
    assert ids[0].tolist() == [int(v) for v in g["sigmoid_ids"]]
    assert w[0].tolist() == [float(v) for v in g["sigmoid_weights"]]


def _ulp32(v):
    v = np.abs(np.asarray(v, dtype=np.float32))
    return (np.nextafter(v, np.float32(np.inf)) - v).astype(np.float64)


def _sigma_mp(l):
    """sigma(l) = 1 / (1 + e^-l) of the float l at 60 decimal digits."""
    import mpmath
    with mpmath.workdps(60):
        return 1 / (1 + mpmath.exp(-mpmath.mpf(float(l))))


def _round_f32_exact(v):
    """The fp32 value nearest to the mpmath value v >= 0 (no ties occur for
    sigma of a nonzero float): a candidate through float64, then the nearest
    of it and its two fp32 neighbours, compared exactly at 60 digits."""
    import mpmath
    c = np.float32(float(v))
    cands = {c, np.nextafter(c, np.float32(np.inf)), np.nextafter(c, np.float32(-np.inf))}
    cands = [f for f in cands if f >= 0]
    with mpmath.workdps(60):
        d = sorted((abs(mpmath.mpf(float(f)) - v), float(f)) for f in cands)
    assert d[0][0] != d[1][0], "tie"
    return np.float32(d[0][1])


def near_midpoint_logits(n_keep=40, n_scan=1 << 22, seed=11):
    """Logits whose sigma, evaluated in float64, lies closest to an fp32
    rounding boundary (the cases a float64 evaluation can round wrongly)."""
    rng = np.random.default_rng(seed)
    l = np.concatenate([rng.uniform(-30, 30, n_scan), rng.standard_normal(n_scan) * 2]).astype(np.float32)
    s64 = 1.0 / (1.0 + np.exp(-l.astype(np.float64)))
    s = s64.astype(np.float32)
    up = np.nextafter(s, np.float32(np.inf)).astype(np.float64)
    dn = np.nextafter(s, np.float32(-np.inf)).astype(np.float64)
    sd = s.astype(np.float64)
    dist = np.minimum(np.abs(s64 - (sd + up) / 2), np.abs(s64 - (sd + dn) / 2)) / s64
    return l[np.argsort(dist)[:n_keep]]


def sigmoid_hard_cases():
    """The fixture of logits whose sigma lies within ~1e-14 (relative) of an
    fp32 rounding boundary (tests/golden/make_sigmoid_hard_cases.py)."""
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "sigmoid_hard_cases.txt")) if not ln.startswith("#")]
    return np.array([int(r[0], 16) for r in rows], dtype=np.uint32).view(np.float32)


def test_sigmoid_correctly_rounded_against_mpmath():
    """The oracle's score is sigma rounded once to the nearest fp32, checked
    against sigma at 60 digits with an exact rounding: random logits over the
    normal, near-one and subnormal ranges of the result, the logits whose
    float64 sigma sits closest to an fp32 rounding boundary in a short scan,
    and the stored hard cases (within ~1e-14 of a boundary: a float64
    evaluation rounds some of them wrongly)."""
    rng = np.random.default_rng(5)
    pts = np.concatenate([rng.uniform(-110, 40, 1500), rng.standard_normal(1500) * 3,
                          rng.uniform(-104, -87, 300), rng.uniform(15, 20, 200),
                          near_midpoint_logits(), sigmoid_hard_cases()]).astype(np.float32)
    got = oracle.sigmoid_f32(pts)
    want = np.array([_round_f32_exact(_sigma_mp(l)) for l in pts], dtype=np.float32)
    bad = np.flatnonzero(got.view(np.uint32) != want.view(np.uint32))
    assert bad.size == 0, [(float(pts[i]), float(got[i]), float(want[i])) for i in bad[:5]]


def test_sigmoid_within_half_ulp_dense_sweep():
    """Over more than a million logits the oracle's score lies within half an
    fp32 spacing of sigma (float64 stands in for the exact value; its error,
    about 2^-52 relative, is covered by a 2^-50 allowance): the property that
    defines a correctly rounded result.  A recipe of a few ulps fails it."""
    rng = np.random.default_rng(9)
    l = np.concatenate([np.linspace(-88, 88, 1 << 20), rng.standard_normal(1 << 18) * 6,
                        np.linspace(-104, -87, 1 << 16)]).astype(np.float32)
    s = oracle.sigmoid_f32(l)
    s64 = 1.0 / (1.0 + np.exp(-l.astype(np.float64)))
    sd = s.astype(np.float64)
    up = np.nextafter(s, np.float32(np.inf)).astype(np.float64) - sd
    dn = sd - np.nextafter(s, np.float32(-np.inf)).astype(np.float64)
    slack = s64 * 2.0 ** -50
    assert np.all(s64 - sd <= up / 2 + slack), float(np.max((s64 - sd) / up))
    assert np.all(sd - s64 <= dn / 2 + slack), float(np.max((sd - s64) / dn))
    assert np.all(np.diff(s[:1 << 20]) >= 0)  # monotone over the sorted sweep


def test_sigmoid_special_values():
    s = oracle.sigmoid_f32(np.array([0.0, -0.0, 17.5, 100.0, -104.0, -200.0, -np.inf, np.inf], np.float32))
    assert s.tolist() == [0.5, 0.5, 1.0, 1.0, 0.0, 0.0, 0.0, 1.0]
    # just below the rounding boundary to 1: 1 - sigma(17) = 4.1e-8 > 2^-25
    assert oracle.sigmoid_f32(np.array([17.0], np.float32))[0] == np.float32(1 - 2.0 ** -24)
    # subnormal results: sigma(-100) = 3.72e-44 = 26.55 * 2^-149 -> 27 * 2^-149
    v = oracle.sigmoid_f32(np.array([-100.0], np.float32))[0]
    assert v == np.float32(27 * 2.0 ** -149) == _round_f32_exact(_sigma_mp(-100.0))


def test_sigmoid_gate_invariants():
    rng = np.random.default_rng(7)
    lg = (rng.standard_normal((8, 896)) * 1.5).astype(np.float32)
    bias = inputs.selection_bias(896)
    ids, w = oracle.route_topk(lg, 16, "sigmoid", bias)
    s = oracle.sigmoid_f32(lg)
    t = (s + bias).astype(np.float32)
    for m in range(8):
        assert _selection_is_valid(t[m], ids[m].tolist())
        ref = s[m, ids[m]].astype(np.float64)
        assert np.max(np.abs(w[m] - ref / ref.sum())) <= 1e-7
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1) <= 16 * 2.0 ** -24)
    # zero bias: sigma is increasing, so (with distinct scores) the softmax ids
    ids0, _ = oracle.route_topk(lg, 16, "sigmoid", np.zeros(896, np.float32))
    idsm, _ = oracle.route_topk(lg, 16, "softmax")
    for m in range(8):
        if len(np.unique(s[m])) == 896:
            assert ids0[m].tolist() == idsm[m].tolist()
    # bias only selects: weights are not the biased scores
    _, w_nr = oracle.route_topk(lg, 16, "sigmoid", bias, renormalize=False)
    assert np.array_equal(w_nr, np.take_along_axis(s, ids, 1))


# ---------------------------------------------------------------- sort


def _brute_sort(ids, N, B):
    """Independent double loop: for each expert in order, scan all flat
    indices in order; pad to B with the sentinel."""
    M, k = ids.shape
    flat = ids.reshape(-1)
    mk = M * k
    cap = mk + min(N, mk) * (B - 1)
    cap = -(-cap // B) * B
    out, blocks = [], []
    for e in range(N):
        run = [f for f in range(mk) if flat[f] == e]
        if not run:
            continue
        padded = run + [mk] * ((-len(run)) % B)
        out += padded
        blocks += [e] * (len(padded) // B)
    ntpp = len(out)
    out += [mk] * (cap - len(out))
    blocks += [-1] * (cap // B - len(blocks))
    return np.array(out, np.int32), np.array(blocks, np.int32), ntpp


@pytest.mark.parametrize("M,k,N,B", [(1, 8, 128, 16), (3, 2, 4, 2), (16, 8, 128, 16),
                                     (7, 16, 896, 16), (64, 8, 128, 64), (5, 3, 7, 1),
                                     (9, 4, 16, 128)])
def test_sort_matches_brute_force(M, k, N, B):
    rng = np.random.default_rng(M * 1000 + k)
    ids = np.stack([rng.permutation(N)[:k] for _ in range(M)]).astype(np.int32)
    st, ex, nt = oracle.moe_sort(ids, N, B)
    bst, bex, bnt = _brute_sort(ids, N, B)
    assert nt == bnt and np.array_equal(st, bst) and np.array_equal(ex, bex)
    # invariants: complete permutation, block counts, owners, alignment
    mk = M * k
    real = st[:nt][st[:nt] != mk]
    assert np.array_equal(np.sort(real), np.arange(mk))
    counts = np.bincount(ids.reshape(-1), minlength=N)
    nblocks = np.bincount(ex[ex >= 0], minlength=N)
    assert np.array_equal(nblocks, -(-counts // B))
    flat = ids.reshape(-1)
    for b in range(nt // B):
        ent = st[b * B:(b + 1) * B]
        assert all(flat[f] == ex[b] for f in ent if f != mk)
    assert nt % B == 0


def test_sort_golden_example():
    g = _golden_kv("sort_example.txt")
    M, k, N, B = (int(g[n][0]) for n in ("M", "k", "N", "B"))
    ids = np.array([int(v) for v in g["topk_ids"]], np.int32).reshape(M, k)
    st, ex, nt = oracle.moe_sort(ids, N, B)
    assert st.tolist() == [int(v) for v in g["sorted_token_ids"]]
    assert ex.tolist() == [int(v) for v in g["expert_ids"]]
    assert nt == int(g["num_tokens_post_padded"][0])


def test_sort_skips_ids_outside_range():
    ids = np.array([[0, -1], [5, 1]], np.int32)  # N = 4: -1 and 5 are masked
    st, ex, nt = oracle.moe_sort(ids, 4, 2)
    assert nt == 4
    assert st[:4].tolist() == [0, 4, 3, 4]
    assert ex[:2].tolist() == [0, 1]


def test_sort_capacity_is_the_worst_case():
    """Every expert used once (count 1 mod B) reaches the bound exactly."""
    for M, k, N, B in [(4, 8, 128, 16), (16, 8, 128, 16), (2, 16, 896, 64), (64, 8, 128, 16)]:
        cap = oracle.sort_capacity(M, k, N, B)
        assert cap % B == 0
        mk = M * k
        worst = mk + min(N, mk) * (B - 1)
        assert cap == -(-worst // B) * B
        if mk <= N:  # all flat indices on distinct experts
            ids = np.arange(mk, dtype=np.int32).reshape(M, k)
            _, _, nt = oracle.moe_sort(ids, N, B)
            assert nt == mk * B and nt <= cap


# ---------------------------------------------------------------- MXFP8


def _e4m3_table():
    """Values of the 254 finite e4m3 codes, straight from the format."""
    codes, vals = [], []
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 0xF, c & 7
        if e == 15 and m == 7:
            continue  # NaN
        v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        codes.append(c)
        vals.append(-v if s else v)
    return np.array(codes), np.array(vals)


def _brute_e4m3(v):
    """Nearest finite code, ties to the even code, saturating, sign kept."""
    codes, vals = _e4m3_table()
    out = np.empty(len(v), np.uint8)
    for i, x in enumerate(v):
        if abs(x) >= 448:
            out[i] = 0x7E | (0x80 if x < 0 else 0)
            continue
        same_sign = (codes >> 7) == (1 if math.copysign(1, x) < 0 else 0)
        c, vv = codes[same_sign], vals[same_sign]
        d = np.abs(vv - x)
        best = np.flatnonzero(d == d.min())
        pick = [b for b in best if c[b] % 2 == 0] if len(best) > 1 else best
        out[i] = c[pick[0]]
    return out


def test_e4m3_encoder_exhaustive_over_bf16_patterns():
    """All 65,536 bf16 patterns (finite ones), scaled by the powers of two the
    quantiser uses, against a brute-force nearest-of-all-codes encoder (run
    on the distinct values only) and torch's own float8_e4m3fn conversion."""
    torch = pytest.importorskip("torch")
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    pats = pats[(pats & 0x7F80) != 0x7F80]  # drop Inf/NaN patterns
    vals = bf16_val(pats)
    checked = 0
    for X in (-127, -100, -20, -8, -3, 0, 3, 8, 20, 100, 127):
        v = np.ldexp(vals, -X)
        v = v[np.abs(v) < 1024.0]
        got = oracle.e4m3_encode_array(v)
        clamped = torch.from_numpy(np.clip(v, -448.0, 448.0)).to(torch.float8_e4m3fn)
        ref = clamped.view(torch.uint8).numpy()
        assert np.array_equal(got, ref), X
        checked += len(v)
    uniq = np.unique(np.ldexp(vals, 0)[np.abs(vals) < 1024.0])
    sample = uniq[:: max(1, len(uniq) // 3000)]
    assert np.array_equal(oracle.e4m3_encode_array(sample), _brute_e4m3(sample))
    assert checked > 100000


def _parse_mx_golden():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "mxfp8_blocks.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] == "case":
                cur = dict(name=parts[1], vals=[], codes=[])
                cases.append(cur)
            elif parts[0] == "scale":
                cur["scale"] = int(parts[1], 16)
            else:
                cur["vals"].append(float(parts[0]))
                cur["codes"].append(int(parts[1], 16))
    return cases


@pytest.mark.parametrize("case", _parse_mx_golden(), ids=lambda c: c["name"])
def test_mxfp8_golden_blocks(case):
    vals = np.zeros(32)
    vals[:len(case["vals"])] = case["vals"]
    x = bf16(vals.reshape(1, 32))
    assert np.array_equal(bf16_val(x)[0], vals), "fixture value not exact in bf16"
    q, s = oracle.mxfp8_quant(x)
    assert s[0, 0] == case["scale"]
    want = np.zeros(32, np.uint8)
    want[:len(case["codes"])] = case["codes"]
    assert q[0].tolist() == want.tolist()


def test_mxfp8_dequant_error_bound_and_edges():
    x = inputs.quant_edge_x(64, 6144)
    q, s = oracle.mxfp8_quant(x)
    xv = bf16_val(x)
    codes, vals = _e4m3_table()
    lut = np.zeros(256)
    lut[codes] = vals
    X = s.astype(np.int64) - 127
    scale = np.repeat(np.ldexp(1.0, X), 32, axis=1)
    deq = lut[q] * scale
    ax = np.abs(xv) / scale
    sat = ax > 448
    # half an e4m3 ulp at the element's binade (quantum 2^-9 below 2^-6)
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -6)))
    half_ulp = np.ldexp(0.5, (e - 3).astype(np.int64))
    assert np.all(np.abs(deq - xv)[~sat] <= (half_ulp * scale)[~sat])
    assert np.all(np.abs(lut[q][sat]) == 448)
    # amax of every nonzero block lies in [2^(X+8), 2^(X+9)) unless clamped
    amax = np.abs(xv).reshape(64, -1, 32).max(2)
    nz = (amax > 0) & (X > -127)
    assert np.all(amax[nz] >= np.ldexp(1.0, X[nz] + 8))
    assert np.all(amax[nz] < np.ldexp(1.0, X[nz] + 9))
    zero_blocks = amax == 0
    assert np.all(s[zero_blocks] == 0)


def test_int32_offset_limit_fixture():
    g = _golden_kv("int32_offset_limit.txt")
    K, limit = int(g["hidden"][0]), int(g["tokens_limit"][0])
    assert (2 ** 31) // K == limit
    assert limit * K < 2 ** 31 <= (limit + 1) * K


# ---------------------------------------------------------------- inputs


def test_inputs_are_deterministic_and_shaped():
    x1, w1 = inputs.router_inputs(4, 6144, 128, 2)
    x2, w2 = inputs.router_inputs(4, 6144, 128, 2)
    assert np.array_equal(x1, x2) and np.array_equal(w1, w2)
    xs = bf16_val(x1)
    ws = bf16_val(w1)
    assert abs(xs.std() - 1.0) < 0.05 and abs(ws.std() - 0.02) < 0.001
    b = inputs.selection_bias(896)
    assert b.min() >= -0.1 and b.max() <= 0.1 and abs(b.mean()) < 0.01
    rows = inputs.scaled_rows(4096)
    assert len(rows) == 40 and len(set(rows.tolist())) == 40
    assert len(inputs.scaled_rows(128)) == 1
