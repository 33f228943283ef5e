"""Error metric used to compare a result against the oracle (test infrastructure).

err = max_i |g_i - r_i| / max(|r_i|, rms(r)), the maximum relative error with
each denominator floored at the root-mean-square of the reference tensor, so
near-zero reference entries do not blow the ratio up.  Pass bars: 1e-5 for
fp32 inputs, 2e-2 for bf16 inputs (state and accumulation in fp32).
"""
from __future__ import annotations

import numpy as np

TOL = {"f32": 1e-5, "bf16": 2e-2}


def rms(r) -> float:
    r = np.asarray(r, dtype=np.float64)
    return float(np.sqrt(np.mean(r * r))) if r.size else 0.0


def floored_rel_err(got, ref, floor: float | None = None) -> float:
    """max |g - r| / max(|r|, floor); floor defaults to rms(ref)."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    if r.size == 0:
        return 0.0
    if not np.all(np.isfinite(g)):
        return float("inf")
    fl = rms(r) if floor is None else float(floor)
    den = np.maximum(np.abs(r), fl)
    den = np.where(den > 0, den, 1.0)
    return float(np.max(np.abs(g - r) / den))


def report(got, ref, floor: float | None = None) -> dict:
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    d = np.abs(g - r)
    nz = np.abs(r) > 0
    return {
        "err": floored_rel_err(g, r, floor),
        "max_abs": float(d.max()) if d.size else 0.0,
        "max_rel_unfloored": float((d[nz] / np.abs(r[nz])).max()) if nz.any() else 0.0,
        "rms_ref": rms(r) if floor is None else float(floor),
    }
