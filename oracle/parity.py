"""Parity criteria between a device result and the oracle (test infrastructure).

* Floating-point outputs stored as bf16: per element
  |g - o| <= 2 * ulp_bf16(max(|o|, rms(o))), and relative L2 <= 2e-3.
  (The per-element ulp is taken no smaller than at the tensor's RMS so that
  elements where routed + shared + residual cancel are not held to an
  unattainable absolute precision.)
* Expert selections: the r-th selected logits must agree within 1e-5
  relative (both zero counts as a tie) at every rank; exact when the logits
  are integers.
"""
from __future__ import annotations

import numpy as np

REL_L2 = 2e-3
ULPS = 2.0
TIE_REL = 1e-5


def ulp_bf16(v) -> np.ndarray:
    """Spacing of the bf16 values around |v|: 2**(e - 7) for |v| in
    [2**e, 2**(e + 1)), and 2**-133 below the smallest normal 2**-126 (bf16
    keeps fp32's exponent range; its subnormals are evenly spaced)."""
    v = np.abs(np.asarray(v, dtype=np.float64))
    _, e = np.frexp(np.where(v > 0, v, 1.0))
    return np.where(v > 0, np.ldexp(1.0, np.maximum(e - 8, -133)), np.ldexp(1.0, -133))


def float_parity(got, ref, rel_l2: float = REL_L2, ulps: float = ULPS):
    """Returns (ok, report) for bf16-stored outputs against oracle values."""
    g = np.asarray(got, dtype=np.float64).ravel()
    o = np.asarray(ref, dtype=np.float64).ravel()
    rms = float(np.sqrt(np.mean(o * o))) if o.size else 0.0
    tol = ulps * ulp_bf16(np.maximum(np.abs(o), rms))
    err = np.abs(g - o)
    worst = int(np.argmax(err - tol)) if o.size else 0
    l2 = float(np.linalg.norm(g - o) / max(np.linalg.norm(o), 1e-300))
    ok = bool(np.all(err <= tol) and (l2 <= rel_l2 or np.linalg.norm(o) == 0))
    rep = (f"rel_l2={l2:.3e} max_err={err.max() if o.size else 0:.3e} "
           f"worst@{worst}: got={g[worst] if o.size else 0:.6g} ref={o[worst] if o.size else 0:.6g} "
           f"tol={tol[worst] if o.size else 0:.3e}")
    return ok, rep


def ids_valid(got_ids, ref_ids, ref_logits, tie_rel: float = TIE_REL) -> bool:
    """GPU selection acceptable against the oracle's fp64 logits."""
    got_ids, ref_ids = list(map(int, got_ids)), list(map(int, ref_ids))
    if got_ids == ref_ids:
        return True
    if len(set(got_ids)) != len(got_ids) or len(got_ids) != len(ref_ids):
        return False
    l = np.asarray(ref_logits, dtype=np.float64)
    if any(e < 0 or e >= l.size for e in got_ids):
        return False
    for a, b in zip(got_ids, ref_ids):
        va, vb = l[a], l[b]
        scale = max(abs(va), abs(vb))
        if scale == 0.0:
            continue
        if abs(va - vb) > tie_rel * scale:
            return False
    return True
