"""Pins of the parity criteria (oracle/parity.py) that every GPU comparison
uses, against library conversions and hand-made cases at their boundaries.

* ulp_bf16 against the spacing of adjacent bf16 values taken from torch's
  bf16 type, normal and subnormal;
* float_parity accepts an error of exactly 2 ulps and rejects one bf16 step
  more, and rejects a relative L2 error just above 2e-3 with every element
  inside its ulp bound;
* ids_valid accepts a swap of two ranks whose logits differ by less than
  1e-5 relative and rejects it at 2e-5, rejects duplicates and out-of-range
  ids, and accepts ties at zero.
"""
import numpy as np
import torch

from oracle import parity as P


def _bf16_values(bits: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def test_ulp_bf16_is_the_spacing_of_adjacent_bf16_values():
    # every positive finite bf16 value below the largest: its spacing upwards
    bits = np.arange(1, 0x7F7F, dtype=np.int64)
    lo, hi = _bf16_values(bits), _bf16_values(bits + 1)
    spacing = hi - lo
    assert np.array_equal(P.ulp_bf16(lo), spacing)
    # values strictly between two neighbours have the same spacing
    mid = lo + spacing * 0.375
    assert np.array_equal(P.ulp_bf16(mid), spacing)
    assert np.array_equal(P.ulp_bf16(-mid), spacing)
    # the subnormal range is evenly spaced at 2**-133
    assert np.all(spacing[lo < 2.0 ** -126] == 2.0 ** -133)
    assert P.ulp_bf16(0.0) == 2.0 ** -133


def test_float_parity_two_ulps_boundary():
    o = np.ones(256)
    g = o.copy()
    g[17] = 1.0 + 2 * 2.0 ** -7          # exactly 2 ulps of 1.0
    ok, _ = P.float_parity(g, o)
    assert ok
    g[17] = 1.0 + 3 * 2.0 ** -7          # one bf16 step more
    ok, _ = P.float_parity(g, o)
    assert not ok
    g = o.copy()
    g[17] = 1.0 - 2 * 2.0 ** -8          # below 1.0 the ulp bound is still the rms's (1.0)
    ok, _ = P.float_parity(g, o)
    assert ok


def test_float_parity_relative_l2_boundary():
    o = np.ones(1024)
    ok, _ = P.float_parity(o * (1 + 1.99e-3), o)
    assert ok
    ok, rep = P.float_parity(o * (1 + 2.01e-3), o)   # every element within 2 ulps (1.56e-2)
    assert not ok, rep


def test_float_parity_floors_the_ulp_at_the_rms():
    o = np.ones(256)
    o[5] = 1e-3                           # a cancelled element: bound set by the rms, not 1e-3
    # rms = 0.998, in [0.5, 1): ulp 2**-8, so the bound is 2**-7 (ulp at 1e-3: 2**-17)
    g = o.copy()
    g[5] = 1e-3 + 0.75 * 2.0 ** -7
    ok, _ = P.float_parity(g, o)
    assert ok
    g[5] = 1e-3 + 1.25 * 2.0 ** -7
    ok, _ = P.float_parity(g, o)
    assert not ok


def test_ids_valid_near_tie_rule():
    logits = np.linspace(10.0, 1.0, 16)
    ref = list(range(8))
    assert P.ids_valid(ref, ref, logits)
    # ranks 7 and 8 within 1e-5 relative: either selection is accepted
    l = logits.copy()
    l[8] = l[7] * (1 - 0.9e-5)
    assert P.ids_valid(list(range(7)) + [8], ref, l)
    l[8] = l[7] * (1 - 2e-5)
    assert not P.ids_valid(list(range(7)) + [8], ref, l)
    # a swap of two ranks inside the selection follows the same rule
    l = logits.copy()
    l[3] = l[2] * (1 - 0.5e-5)
    assert P.ids_valid([0, 1, 3, 2, 4, 5, 6, 7], ref, l)
    l[3] = l[2] * (1 - 2e-5)
    assert not P.ids_valid([0, 1, 3, 2, 4, 5, 6, 7], ref, l)


def test_ids_valid_rejects_duplicates_and_out_of_range():
    logits = np.zeros(16)                 # every logit ties at zero
    ref = list(range(8))
    assert P.ids_valid([1, 0, 2, 3, 4, 5, 6, 7], ref, logits)     # ties at zero accepted
    assert not P.ids_valid([0, 0, 2, 3, 4, 5, 6, 7], ref, logits)
    assert not P.ids_valid([0, 1, 2, 3, 4, 5, 6, 16], ref, logits)
    assert not P.ids_valid([0, 1, 2, 3, 4, 5, 6, -1], ref, logits)
    assert not P.ids_valid([0, 1, 2, 3, 4, 5, 6], ref, logits)
