"""Seeded synthetic inputs for the MoE decode routing path.

This module only draws numbers and rounds them to the storage types the
routing path reads (bf16 activations and gate weights, fp32 selection bias).
It holds none of the routing arithmetic (no GEMV, gating, sort or quant),
so both the CUDA path's tests and the CPU oracle can take their inputs from
it without sharing any step of the method.

Recipe (the same bytes on every machine, numpy only):

* Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
  number generators", OOPSLA 2014) used counter-style: draw ``i`` of a stream
  is ``mix64(key + (i + 1) * 0x9E3779B97F4A7C15)`` with the published
  finaliser.  A stream's key is ``mix64`` of ``(seed, config id, tensor tag)``
  packed into one 64-bit word.
* Uniform (0, 1): the top 53 bits of a draw, plus one half, times 2**-53.
* Normal: Box-Muller on consecutive uniform pairs, in float64.
* bf16: float64 -> float32 (round to nearest even) -> bf16 (round to nearest
  even on the upper 16 bits).

Shapes and distributions follow the workloads the routing pages describe
(MiniMax-M3 style routing: N = 128 experts, hidden K = 6144, top-8; Kimi-K3
style routing: N = 896, K = 3584, top-16, sigmoid scores with a selection
bias): x ~ N(0, 1), gate W ~ N(0, 0.02), bias ~ U(-0.1, 0.1).
"""

from __future__ import annotations

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(config_id: int, tag: int, seed: int = 0) -> int:
    """64-bit key of the stream for one tensor of one workload."""
    packed = ((seed & 0xFFFFFF) << 40) | ((config_id & 0xFFFFF) << 20) | (tag & 0xFFFFF)
    return int(_mix64(np.array([packed], dtype=np.uint64))[0])


def draws_u64(key: int, n: int, offset: int = 0) -> np.ndarray:
    """Draws ``offset .. offset + n - 1`` of the SplitMix64 stream ``key``."""
    i = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        state = np.uint64(key) + i * _GAMMA
    return _mix64(state)


def uniform01(key: int, n: int, offset: int = 0) -> np.ndarray:
    """n float64 values in the open interval (0, 1)."""
    u = draws_u64(key, n, offset) >> np.uint64(11)
    return (u.astype(np.float64) + 0.5) * (2.0 ** -53)


def normal(key: int, n: int) -> np.ndarray:
    """n float64 N(0, 1) values by Box-Muller."""
    pairs = (n + 1) // 2
    u = uniform01(key, 2 * pairs)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * pairs, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return z[:n]


def f64_to_bf16_bits(a) -> np.ndarray:
    """float64 -> bf16 bit patterns (uint16), via float32, both steps RNE."""
    f32 = np.ascontiguousarray(np.asarray(a, dtype=np.float64).astype(np.float32))
    bits = f32.view(np.uint32).astype(np.uint64)
    rounded = (bits + np.uint64(0x7FFF) + ((bits >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return rounded.astype(np.uint16).reshape(f32.shape)


def bf16_bits_to_f32(b) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact)."""
    b = np.ascontiguousarray(np.asarray(b, dtype=np.uint16))
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


# Tensor tags inside one workload's key space.
TAG_X, TAG_W, TAG_BIAS, TAG_ROWS, TAG_EDGE, TAG_VARIANT = 1, 2, 3, 4, 5, 6
TAG_RMS, TAG_NORMW = 7, 8
TAG_SH_CODE, TAG_SH_SCALE = 9, 10


def normal_bf16(shape, std: float, config_id: int, tag: int, seed: int = 0) -> np.ndarray:
    n = int(np.prod(shape))
    z = normal(stream_key(config_id, tag, seed), n) * std
    return f64_to_bf16_bits(z).reshape(shape)


def uniform_f32(shape, lo: float, hi: float, config_id: int, tag: int, seed: int = 0) -> np.ndarray:
    n = int(np.prod(shape))
    u = uniform01(stream_key(config_id, tag, seed), n)
    return (lo + (hi - lo) * u).astype(np.float32).reshape(shape)


def fisher_yates(n: int, key: int) -> np.ndarray:
    """A seeded uniform permutation of 0..n-1 (Durstenfeld's in-place shuffle)."""
    perm = np.arange(n, dtype=np.int64)
    u = uniform01(key, max(n - 1, 0))
    for step, i in enumerate(range(n - 1, 0, -1)):
        j = int(u[step] * (i + 1))
        perm[i], perm[j] = perm[j], perm[i]
    return perm


# ---------------------------------------------------------------------------
# Workloads.  Each returns numpy arrays: x and W as bf16 bits (uint16),
# bias as float32.  ``variant`` selects an independent draw of the same
# workload (used to rotate copies through memory and to vary launches).
# ---------------------------------------------------------------------------

def router_inputs(M: int, K: int, N: int, config_id: int, seed: int = 0, variant: int = 0):
    """x [M, K] ~ N(0, 1) and gate W [N, K] ~ N(0, 0.02), both bf16 bits."""
    vtag = variant << 8
    x = normal_bf16((M, K), 1.0, config_id, TAG_X | vtag, seed)
    w = normal_bf16((N, K), 0.02, config_id, TAG_W | vtag, seed)
    return x, w


def selection_bias(N: int, config_id: int = 3, seed: int = 0) -> np.ndarray:
    """Per-expert selection bias ~ U(-0.1, 0.1), float32 [N]."""
    return uniform_f32((N,), -0.1, 0.1, config_id, TAG_BIAS, seed)


def scaled_rows(M: int, config_id: int = 4, seed: int = 0) -> np.ndarray:
    """Rows of x scaled by 50: max(1, M // 100) rows from a seeded shuffle."""
    n = max(1, M // 100)
    perm = fisher_yates(M, stream_key(config_id, TAG_ROWS, seed))
    return np.sort(perm[:n])


def prefill_x(M: int, K: int, config_id: int = 4, seed: int = 0, variant: int = 0) -> np.ndarray:
    """x [M, K] ~ N(0, 1) with 1 % of its rows scaled by 50 (bf16 bits)."""
    z = normal(stream_key(config_id, TAG_X | (variant << 8), seed), M * K).reshape(M, K)
    z[scaled_rows(M, config_id, seed)] *= 50.0
    return f64_to_bf16_bits(z)


def norm_inputs(M: int, K: int, config_id: int = 6, seed: int = 0, variant: int = 0):
    """Un-normalised residual rows, their rstd and a Gemma-style norm weight.

    Row m has its own magnitude a_m ~ U(0.5, 8): sres[m] = bf16(a_m * z),
    z ~ N(0, 1); rstd[m] = float32(1 / a_m) stands for what the norm in
    front of the router publishes (the router only multiplies by it, so any
    positive value of that size exercises the same arithmetic); the norm
    weight g ~ N(0, 0.1) in bf16 (offsets around 0, applied as 1 + g by a
    Gemma RMSNorm).  Returns (sres bf16 bits [M, K], rstd float32 [M],
    g bf16 bits [K]).
    """
    vtag = variant << 8
    amp = 0.5 + 7.5 * uniform01(stream_key(config_id, TAG_RMS | vtag, seed), M)
    z = normal(stream_key(config_id, TAG_X | vtag, seed), M * K).reshape(M, K)
    sres = f64_to_bf16_bits(z * amp[:, None])
    rstd = (1.0 / amp).astype(np.float32)
    g = normal_bf16((K,), 0.1, config_id, TAG_NORMW | vtag, seed)
    return sres, rstd, g


def shared_expert_weights(I: int, K: int, config_id: int = 7, seed: int = 0, variant: int = 0):
    """Synthetic MXFP8 gate/up weights of a shared expert: E4M3 codes
    [2I, K] (rows [0, I) gate, [I, 2I) up) and E8M0 scale bytes [2I, K/32].

    Codes are drawn as bit fields: a random sign, an exponent field uniform
    in 4..11 and a mantissa uniform in 0..7 (magnitudes 2^-3 .. 30, never the
    NaN code); scale bytes 127 + X with X uniform in -12..-8, so that a
    weight is about 3e-5 .. 0.12, the size of the gate weights here.
    """
    vtag = variant << 8
    d = draws_u64(stream_key(config_id, TAG_SH_CODE | vtag, seed), 2 * I * K)
    sign = (d & np.uint64(1)).astype(np.uint8) << 7
    expo = (4 + ((d >> np.uint64(8)) % np.uint64(8))).astype(np.uint8)
    mant = ((d >> np.uint64(16)) & np.uint64(7)).astype(np.uint8)
    codes = (sign | (expo << 3) | mant).reshape(2 * I, K)
    ds = draws_u64(stream_key(config_id, TAG_SH_SCALE | vtag, seed), 2 * I * (K // 32))
    scale = (127 - 12 + (ds % np.uint64(5))).astype(np.uint8).reshape(2 * I, K // 32)
    return codes, scale


def tied_gate(w: np.ndarray, pairs=((10, 11), (50, 51))) -> np.ndarray:
    """Copy gate row a onto row b for each (a, b): forced exact logit ties."""
    w = w.copy()
    for a, b in pairs:
        w[b] = w[a]
    return w


# Largest bf16 strictly below 448 (the e4m3 maximum) is 446; the next above is 450.
_EDGE_AMAX = (446.0, 448.0, 450.0)


def quant_edge_x(M: int, K: int, config_id: int = 5, seed: int = 0) -> np.ndarray:
    """x [M, K] ~ N(0, 1) with 32-element blocks replaced by quantiser edge cases.

    Block kinds (row r, block b of 32 along K), placed row by row from row 0:
    all zeros; negative zeros; random bf16 subnormals; a subnormal block whose
    amax forces the lowest scale; for k in (-10, 0, 5) blocks whose amax is
    446 * 2**k, 448 * 2**k and 450 * 2**k (just under, at and just over the
    e4m3 maximum times a power of two); an exact power of two; the largest
    finite bf16; and a block mixing huge and tiny magnitudes.
    """
    assert K % 32 == 0
    x = normal_bf16((M, K), 1.0, config_id, TAG_X, seed).copy()
    rng_key = stream_key(config_id, TAG_EDGE, seed)
    draws = draws_u64(rng_key, 4096)
    cursor = [0]

    def take(n):
        out = draws[cursor[0]:cursor[0] + n]
        cursor[0] += n
        return out

    blocks = []
    blocks.append(np.zeros(32, dtype=np.uint16))                     # all +0
    blocks.append(np.full(32, 0x8000, dtype=np.uint16))              # all -0
    sub = (take(32) & np.uint64(0x807F)).astype(np.uint16)           # sign + mantissa only
    sub[sub & 0x7F == 0] |= 1
    blocks.append(sub)                                               # subnormals
    tiny = np.zeros(32, dtype=np.uint16)
    tiny[5] = 0x0001                                                 # smallest subnormal
    tiny[9] = 0x8003
    blocks.append(tiny)
    base = normal(rng_key ^ 0x5555, 32 * 16)
    bi = 0
    for k in (-10, 0, 5):
        for amax in _EDGE_AMAX:
            v = base[bi * 32:(bi + 1) * 32] * (2.0 ** k)
            v[(bi * 7) % 32] = (-1.0 if bi % 2 else 1.0) * amax * 2.0 ** k
            blocks.append(f64_to_bf16_bits(v))
            bi += 1
    p2 = base[bi * 32:(bi + 1) * 32].copy()
    p2[3] = 2.0 ** 7                                                 # amax exactly 128
    blocks.append(f64_to_bf16_bits(p2))
    bi += 1
    big = f64_to_bf16_bits(base[bi * 32:(bi + 1) * 32] * 1e30)
    big[0] = 0x7F7F                                                  # largest finite bf16
    blocks.append(big)
    bi += 1
    mix = base[bi * 32:(bi + 1) * 32] * 1e-3
    mix[17] = -3.0e4
    blocks.append(f64_to_bf16_bits(mix))

    per_row = K // 32
    for i, blk in enumerate(blocks):
        r, b = divmod(i * 5, per_row)
        r = r % M
        x[r, b * 32:(b + 1) * 32] = blk
    return x


CONFIGS = {
    1: dict(name="decode M=1, K=6144, N=128, softmax top-8, block 16", K=6144, N=128, topk=8,
            block=16, scoring="softmax", Ms=(1,)),
    2: dict(name="decode buckets M=2..64, K=6144, N=128, softmax top-8, block 16", K=6144, N=128,
            topk=8, block=16, scoring="softmax", Ms=(2, 4, 8, 16, 32, 64)),
    3: dict(name="large-expert routing K=3584, N=896, sigmoid+bias top-16, block 16", K=3584,
            N=896, topk=16, block=16, scoring="sigmoid", Ms=(1, 8, 16, 32)),
    4: dict(name="extended rows M=128..512 and prefill sort+quant M=4096, block 64", K=6144,
            N=128, topk=8, block=64, scoring="softmax", Ms=(128, 256, 512), prefill_M=4096),
    5: dict(name="adversarial M=64, K=6144, N=128, top-8: skew, ties, quant edges", K=6144,
            N=128, topk=8, block=16, scoring="softmax", Ms=(64,)),
    6: dict(name="route on the norm's scale: residual rows + rstd + Gemma norm weight, M=1..64, "
                 "K=6144, N=128, softmax top-8, block 16", K=6144, N=128, topk=8, block=16,
            scoring="softmax", Ms=(1, 2, 4, 8, 16, 32, 64)),
}
