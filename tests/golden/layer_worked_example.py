"""Writes layer_worked_example.txt: a whole MoE layer small enough to work out
by hand, with the expected values evaluated from their closed forms.

This script imports neither the oracle nor the library: every expected value
below is the closed form written in the comments, evaluated with the standard
library, and rounded to bf16 by the definition of round-to-nearest-even on 8
significant bits. Run it to regenerate the fixture:

    python tests/golden/layer_worked_example.py

The layer (H = 256, E = 8 experts, top-2, expert width I = 256, shared width
256, bf16 weights, eps = 1e-6); every weight not listed is zero:

  x[0] = 1, x[1] = 2
  residual[h] = (-0.75, -0.25, 0.25, 0.75)[h % 4], except residual[3] = 138/4096
  router   W_r[e, 0] = c_e,  c = (0.5, 1, -1, 2, 0.25, 1, -2, 0)
  expert e G_e[0, 0] = 1;  U_e[0, 1] = (e + 1)/8;  D_e[e, 0] = 1, D_e[e + 8, 0] = -1/2
  shared   G_s[0, 0] = 1;  U_s[0, 1] = 1/4;  D_s[3, 0] = 11/32, D_s[20, 0] = 1,
           D_s[21, 0] = -1;  w_sg[1] = -1/2
  w_norm[h] = 1 + (h % 2)/2

Derivation (s1 = sigma(1) = 1/(1 + e^-1); silu(1) = s1):
  logits = c. Top-2 by value descending, ties to the lower index: expert 3
  (logit 2), then experts 1 and 5 tie at 1 and expert 1 wins. ids = (3, 1).
  Softmax over the two selected logits (2, 1): w = (s1, 1 - s1).
  Expert 3: g0 = 1, u0 = (4/8)*2 = 1, h0 = s1; y_3 = s1 (e_3 - e_11 / 2).
  Expert 1: g0 = 1, u0 = (2/8)*2 = 1/2, h0 = s1/2; y_1 = s1/2 (e_1 - e_9 / 2).
  routed = s1*y_3 + (1 - s1)*y_1:
    routed[3] = s1^2, routed[11] = -s1^2/2,
    routed[1] = s1 (1 - s1)/2, routed[9] = -s1 (1 - s1)/4.
  Shared: g0 = 1, u0 = (1/4)*2 = 1/2, h0 = s1/2; y_s = s1/2 (11/32 e_3 + e_20 - e_21);
    gate sigma(w_sg . x) = sigma(-1) = 1 - s1;
    shared = (1 - s1) s1/2 (11/32 e_3 + e_20 - e_21).
  Fold: t = bf16(bf16(routed) + bf16(shared)); sum = bf16(t + residual);
    r = 1/sqrt(mean(sum^2) + eps); y = bf16(sum * r * w_norm).
  Without a shared expert (the 2-input branch): sum = bf16(bf16(routed) + residual).
  Row 3 makes the rounding of routed to bf16 before the fold visible: with the
  shared expert, bf16(shared[3]) = 138/4096 and bf16(s1^2) + 138/4096 lies above
  the midpoint 291/512 while s1^2 + 138/4096 lies below it, so t[3] is 146/256
  only if routed is rounded first (145/256 otherwise); without the shared
  expert, residual[3] = 138/4096 does the same for sum[3].
"""
import math
import os

H = 256
C = (0.5, 1.0, -1.0, 2.0, 0.25, 1.0, -2.0, 0.0)
RES3 = 138.0 / 4096.0
EPS = 1e-6


def bf16(v: float) -> float:
    """Round-to-nearest-even on 8 significant bits (normal range only, which
    is all this example needs)."""
    if v == 0.0:
        return 0.0
    e = math.floor(math.log2(abs(v)))
    if 2.0 ** e > abs(v):          # guard log2 rounding at binade edges
        e -= 1
    if 2.0 ** (e + 1) <= abs(v):
        e += 1
    q = 2.0 ** (e - 7)
    return round(v / q) * q        # v / q is exact; round() is half-to-even


def residual():
    r = [(-0.75, -0.25, 0.25, 0.75)[h % 4] for h in range(H)]
    r[3] = RES3
    return r


def w_norm():
    return [1.0 + 0.5 * (h % 2) for h in range(H)]


def expected(with_shared: bool):
    s1 = 1.0 / (1.0 + math.exp(-1.0))
    routed = [0.0] * H
    routed[3] = s1 * s1
    routed[11] = -s1 * s1 / 2
    routed[1] = s1 * (1 - s1) / 2
    routed[9] = -s1 * (1 - s1) / 4
    shared = [0.0] * H
    if with_shared:
        shared[3] = (1 - s1) * s1 / 2 * (11.0 / 32.0)
        shared[20] = (1 - s1) * s1 / 2
        shared[21] = -(1 - s1) * s1 / 2
    routed16 = [bf16(v) for v in routed]
    shared16 = [bf16(v) for v in shared]
    res = residual()
    if with_shared:
        t = [bf16(a + b) for a, b in zip(routed16, shared16)]
    else:
        t = routed16
    s = [bf16(a + b) for a, b in zip(t, res)]
    r = 1.0 / math.sqrt(sum(v * v for v in s) / H + EPS)
    wn = w_norm()
    y = [bf16(v * r * w) for v, w in zip(s, wn)]
    # no y value may sit within 1e-6 of a bf16 spacing from a rounding
    # midpoint, so that the order of the two fp64 products cannot change its
    # bf16 rounding
    for v, w in zip(s, wn):
        z = v * r * w
        if z != 0.0:
            e = math.floor(math.log2(abs(z)))
            q = 2.0 ** (e - 7)
            frac = abs(z / q) - math.floor(abs(z / q))
            assert abs(frac - 0.5) > 1e-6, z
    return {"ids": [3.0, 1.0], "w": [s1, 1 - s1], "routed": routed, "shared": shared,
            "routed_bf16": routed16, "shared_bf16": shared16, "sum": s, "y": y}


def main():
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "layer_worked_example.txt")
    lines = ["# Whole MoE layer worked by hand: inputs, derivation and closed forms are in",
             "# layer_worked_example.py (this file is its output). Keys with the suffix _2in",
             "# are the same layer without a shared expert (2-input residual norm).",
             "# Values are decimal float64 with 17 significant digits."]
    for suffix, with_shared in (("", True), ("_2in", False)):
        ex = expected(with_shared)
        for key in ("ids", "w", "routed", "shared", "routed_bf16", "shared_bf16", "sum", "y"):
            if suffix and key in ("shared", "shared_bf16"):
                continue
            lines.append(key + suffix + " " + " ".join(repr(float(v)) for v in ex[key]))
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
