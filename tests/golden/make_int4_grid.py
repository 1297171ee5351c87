"""Writes int4_grid.json: a hand-derived int4 example (no oracle call).

Two output rows, 64 inputs (two groups of 32).  Every group's weights lie on
a grid of step s, and the group's range [min(0, min w), max(0, max w)] is
exactly 15 steps wide, so the quantiser must find scale s, zero point
z = -min / s and codes q = w / s + z with no rounding at all; dequantising
gives the weights back bit for bit.
"""
import json
import os

groups = {
    # (output row, group): (step s, integer multipliers k of the 32 weights)
    (0, 0): (0.125, [k for k in range(-8, 8)] * 2),     # min -1, max 0.875 -> z 8
    (0, 1): (0.125, [k for k in range(0, 16)] * 2),     # min 0 (clamped), max 1.875 -> z 0
    (1, 0): (0.125, [-k for k in range(0, 16)] * 2),    # min -1.875, max 0 -> z 15
    (1, 1): (0.0625, [k for k in range(-8, 8)] * 2),    # min -0.5, max 0.4375 -> z 8
}
W = [[0.0, 0.0] for _ in range(64)]
scales = [[0.0, 0.0], [0.0, 0.0]]
zeros = [[0, 0], [0, 0]]
codes = [[0] * 64, [0] * 64]
for (o, g), (s, ks) in groups.items():
    z = -min(0, min(ks))
    scales[o][g] = s
    zeros[o][g] = z
    for j, k in enumerate(ks):
        W[32 * g + j][o] = k * s
        codes[o][32 * g + j] = k + z
out = {"source": "hand-derived from the grouped asymmetric int4 definition "
                  "(model.fir header: transpose to [output,input], grouped asymmetric int4; "
                  "group 32, fp32 scale, 4-bit zero point)",
       "W_in_out": W, "scales": scales, "zeros": zeros, "codes": codes}
with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "int4_grid.json"), "w") as f:
    json.dump(out, f, indent=0)
