"""Writes sigmoid_hard_cases.txt: fp32 logits whose sigmoid lies closest to an
fp32 rounding boundary (a midpoint between two adjacent fp32 values).

These are the inputs on which an evaluation that is merely accurate (float64,
an error near 2^-52) may round to the wrong fp32 neighbour, so they test that
a score is correctly rounded.  Only the INPUTS are stored; the expected scores
are computed by the tests at 60 digits.  The scan evaluates sigma in float64
for 2^30 seeded random logits and keeps the closest cases (distance relative
to sigma, as estimated in float64).  Run from the repository root:

    python tests/golden/make_sigmoid_hard_cases.py
"""

import os

import numpy as np

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "sigmoid_hard_cases.txt")
CHUNK, CHUNKS, KEEP = 1 << 24, 64, 64


def main():
    rng = np.random.default_rng(20261203)
    best_l = np.empty(0, np.float32)
    best_d = np.empty(0, np.float64)
    for c in range(CHUNKS):
        if c % 2 == 0:
            l = rng.uniform(-18, 18, CHUNK).astype(np.float32)
        else:
            l = (rng.standard_normal(CHUNK) * 3).astype(np.float32)
        s64 = 1.0 / (1.0 + np.exp(-l.astype(np.float64)))
        s = s64.astype(np.float32)
        sd = s.astype(np.float64)
        up = np.nextafter(s, np.float32(np.inf)).astype(np.float64)
        dn = np.nextafter(s, np.float32(-np.inf)).astype(np.float64)
        d = np.minimum(np.abs(s64 - (sd + up) / 2), np.abs(s64 - (sd + dn) / 2)) / s64
        sel = np.argpartition(d, KEEP)[:KEEP]
        best_l = np.concatenate([best_l, l[sel]])
        best_d = np.concatenate([best_d, d[sel]])
        _, first = np.unique(best_l.view(np.uint32), return_index=True)  # a logit drawn twice counts once
        best_l, best_d = best_l[first], best_d[first]
        keep = np.argsort(best_d)[:KEEP]
        best_l, best_d = best_l[keep], best_d[keep]
    with open(OUT, "w") as f:
        f.write("# fp32 logits (bit pattern, value) whose sigmoid lies closest to an fp32 rounding\n")
        f.write("# boundary; distance = |sigma - midpoint| / sigma as estimated in float64.\n")
        f.write("# Written by make_sigmoid_hard_cases.py (2^30 seeded random logits scanned).\n")
        for l, d in zip(best_l, best_d):
            f.write(f"{int(np.float32(l).view(np.uint32)):08x} {float(l):.9g} {d:.3e}\n")


if __name__ == "__main__":
    main()
