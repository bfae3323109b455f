"""Pins of the oracle's float expert modes and gate function, against brute
force on tiny integer inputs and closed forms (no GPU):

* the diagnostic float mode (dequantised weights x unquantised activations)
  equals an exact integer computation when the Q8_0 scales are 1;
* the tensor-core (fp16) mode equals the float mode on fp16-exact inputs up
  to the fp16 rounding of h, within that rounding's bound;
* sigmoid and silu against their closed forms.
"""
import math

import numpy as np
import torch

import gen
from oracle import moe as M

H, I = 64, 32


def _unit_scale_rows(rows, k, seed, lo, hi):
    """Integer weights [rows, k] whose 32-blocks each hold one +-127 (at
    element 0), so Q8_0 encodes them with d = 1 exactly and codes = the
    integers themselves."""
    rng = np.random.default_rng(seed)
    w = rng.integers(lo, hi + 1, (rows, k)).astype(np.float32)
    w[:, ::32] = np.where(rng.integers(0, 2, (rows, k // 32)) > 0, 127.0, -127.0)
    return w


def _tiny_expert(seed):
    wg = _unit_scale_rows(I, H, seed, -2, 2)
    wu = _unit_scale_rows(I, H, seed + 1, -2, 2)
    wd = _unit_scale_rows(H, I, seed + 2, -2, 2)
    x = np.random.default_rng(seed + 3).integers(-1, 2, H).astype(np.float64)
    x[::32] = 0.0                       # the +-127 columns do not contribute
    enc = [gen.encode_q8_0(torch.from_numpy(w)).numpy() for w in (wg, wu, wd)]
    return wg, wu, wd, x, enc


def test_float_mode_equals_integer_brute_force():
    for seed in range(4):
        wg, wu, wd, x, (g8, u8, d8) = _tiny_expert(10 * seed)
        f = M.expert_ffn_float("q8_0", g8, u8, d8, x)
        gi = [int(sum(int(wg[i, k]) * int(x[k]) for k in range(H))) for i in range(I)]
        ui = [int(sum(int(wu[i, k]) * int(x[k]) for k in range(H))) for i in range(I)]
        assert f["g"].tolist() == gi and f["u"].tolist() == ui
        h = [gi[i] / (1.0 + math.exp(-gi[i])) * ui[i] for i in range(I)]
        assert np.allclose(f["h"], h, rtol=1e-13, atol=1e-13)
        y = [math.fsum(float(wd[j, i]) * h[i] for i in range(I)) for j in range(H)]
        assert np.allclose(f["y"], y, rtol=1e-12, atol=1e-9)


def test_fp16_mode_is_the_float_mode_up_to_the_rounding_of_h():
    for seed in range(4):
        wg, wu, wd, x, (g8, u8, d8) = _tiny_expert(100 + 10 * seed)
        f = M.expert_ffn_float("q8_0", g8, u8, d8, x)
        t = M.expert_ffn_fp16("q8_0", g8, u8, d8, x)
        # weights and x are small integers: exact in fp16, so g and u agree exactly
        assert np.array_equal(t["g"], f["g"]) and np.array_equal(t["u"], f["u"])
        assert np.max(np.abs(f["h"])) < 65504                # h stays in the fp16 range
        # y differs only through h's rounding to fp16: |dh| <= |h| * 2^-11
        bound = np.abs(wd.astype(np.float64)) @ (np.abs(f["h"]) * 2.0 ** -11)
        assert np.all(np.abs(t["y"] - f["y"]) <= bound + 1e-9)
        assert np.any(t["y"] != f["y"])                       # the rounding does show


def test_sigmoid_and_silu_closed_forms():
    z = np.linspace(-30.0, 30.0, 601)
    s = M.sigmoid(z)
    assert M.sigmoid(0.0) == 0.5
    assert np.allclose(s + M.sigmoid(-z), 1.0, rtol=0, atol=1e-15)
    assert abs(M.sigmoid(math.log(3.0)) - 0.75) < 1e-15
    assert np.allclose(s, np.exp(z) / (1.0 + np.exp(z)), rtol=1e-14, atol=0)
    assert np.all(np.diff(s) > 0)
    assert np.allclose(M.silu(z), z * s, rtol=1e-14, atol=1e-300)
    assert M.silu(0.0) == 0.0
