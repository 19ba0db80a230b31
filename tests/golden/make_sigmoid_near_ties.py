"""Writes sigmoid_near_ties.txt: pairs of (logit, selection bias) whose fp64 routing keys
key = sigmoid(u) + b differ by 0, 1 or 2 units in the last place.

Routing ("DeepSeek MoE：从v1到v3的演进", DeepSeek-v3: sigmoid gate, selection-only bias) ranks
experts by key = sigmoid(u) + b. The fp64 oracle rounds each step; a token whose K-th and
(K+1)-th keys differ by one or two fp64 units sits on the finest decision the oracle makes.
These inputs let the GPU tests check that such decisions come out the same on both sides.

Construction (inputs only, every key computed by the oracle's own fp64 sigmoid):
  u runs over consecutive fp32 values in [-0.504, -0.5), so s = sigmoid(u) lies in [0.25, 0.5)
  where one fp64 unit is 2^-54. Write s = q + r with q a multiple of 2^-34 and 0 <= r < 2^-34
  (exact in fp64). For two logits a, b whose remainders differ by at most two units, the bias
  D = q_a - q_b is a multiple of 2^-34 below 2^-10, hence an exact fp32 number, and
  key_b = s_b + D = q_a + r_b is exact in fp64, so key_a - key_b = r_a - r_b exactly.
Each output line: u_a u_b D d, the fp32 values as hex floats and d = (key_a - key_b) / 2^-54.

Run from the repository root: python tests/golden/make_sigmoid_near_ties.py
"""
from __future__ import annotations

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "sigmoid_near_ties.txt")
GRID = 2.0 ** -34
ULP = 2.0 ** -54
PER_D = 24  # pairs kept for each difference d in -2..2


def main():
    lo = np.float32(-0.504)
    hi = np.float32(-0.5)
    u = np.arange(lo.view(np.int32), hi.view(np.int32), -1, dtype=np.int32).view(np.float32)
    u = u[(u >= lo) & (u < hi)]
    s = oracle.scores(u.astype(np.float64)[None, :], "sigmoid")[0]
    assert (s >= 0.25).all() and (s < 0.5).all()
    q = np.floor(s / GRID) * GRID
    r = s - q
    order = np.argsort(r, kind="stable")
    rs = r[order]
    rng = np.random.default_rng(0)
    found = {d: [] for d in range(-2, 3)}
    # candidate partners: the next few entries in remainder order
    for step in range(1, 4):
        i = np.arange(len(rs) - step)
        j = i + step
        diff = np.rint((rs[i] - rs[j]) / ULP).astype(np.int64)
        for a_pos, b_pos, d in zip(i[np.abs(diff) <= 2], j[np.abs(diff) <= 2], diff[np.abs(diff) <= 2]):
            a, b = order[a_pos], order[b_pos]
            if rng.random() < 0.5:  # either logit may be the biased one
                a, b, d = b, a, -d
            found[int(d)].append((a, b))
    lines = ["# Near-tie routing keys: u_a u_b D d (hex floats; fp32 values). key_a = sigmoid(u_a),",
             "# key_b = sigmoid(u_b) + D, both in fp64 as the oracle computes them;",
             "# d = (key_a - key_b) / 2^-54 exactly. Written by make_sigmoid_near_ties.py (oracle only)."]
    for d in range(-2, 3):
        pairs = found[d]
        pick = rng.choice(len(pairs), size=min(PER_D, len(pairs)), replace=False)
        for k in sorted(pick):
            a, b = pairs[k]
            D = np.float32(q[a] - q[b])
            assert float(D) == q[a] - q[b] and abs(float(D)) < 2.0 ** -10
            ka = s[a]
            kb = s[b] + np.float64(D)
            assert kb == q[a] + r[b] and (ka - kb) / ULP == d
            lines.append(f"{float(u[a]).hex()} {float(u[b]).hex()} {float(D).hex()} {d}")
    with open(OUT, "w") as fh:
        fh.write("\n".join(lines) + "\n")
    print(OUT, {d: len(v) for d, v in found.items()})


if __name__ == "__main__":
    main()
