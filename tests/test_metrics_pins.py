"""Pins of the parity checker (oracle/metrics.py) on hand-computed cases.

Every GPU parity test passes through floored_rel_err, so it is pinned here against
values worked out by hand, independent of its own code:

  err = max_i |g_i - r_i| / max(|r_i|, rms(r)),  rms(r) = sqrt(mean(r^2))

(the reading of "max relative error" taken for this path: a relative error whose
denominator is floored at the reference tensor's root-mean-square, so that entries
of the reference near zero do not dominate).  Each case is chosen so that a
plausible slip fails it: the mean in place of the max, the floor at max|r| or at
mean|r| in place of the rms, the rms without its square root, a dropped abs, the
non-finite guard dropped.  The module under test can be replaced through the
SSM_METRICS_PATH environment variable (used by the planted-mistake tests).
"""
import importlib.util
import math
import os

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _load():
    path = os.environ.get("SSM_METRICS_PATH", os.path.join(ROOT, "oracle", "metrics.py"))
    spec = importlib.util.spec_from_file_location("metrics_under_test", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


M = _load()


def test_rms_by_hand():
    # sqrt((9 + 16) / 2) = sqrt(12.5)
    assert M.rms([3.0, -4.0]) == pytest.approx(math.sqrt(12.5), rel=1e-15)
    assert M.rms([]) == 0.0


def test_max_not_mean_and_floor_absorbs_zero_reference():
    # rms(ref) = sqrt((1 + 4 + 0 + 1e-6) / 4); the entry with ref 0 is divided by the
    # rms, not by 0; the worst ratio is entry 0's 0.1 / rms
    ref = np.array([1.0, -2.0, 0.0, 1e-3])
    got = np.array([1.1, -2.0, 0.01, 1e-3])
    rms = math.sqrt((1.0 + 4.0 + 0.0 + 1e-6) / 4.0)
    want = max(0.1 / max(1.0, rms), 0.0, 0.01 / rms, 0.0)
    assert want == pytest.approx(0.1 / rms)
    assert M.floored_rel_err(got, ref) == pytest.approx(want, rel=1e-12)
    # the mean of the ratios would be about a quarter of this
    assert M.floored_rel_err(got, ref) > 0.08


def test_floor_is_the_rms_not_the_largest_entry():
    # rms = sqrt((100 + 3 * 0.01) / 4) = sqrt(25.0075); entry 3 differs by 0.1 and its
    # own magnitude (0.1) is below the floor: err = 0.1 / sqrt(25.0075) = 0.019997
    # (a floor at max|r| = 10 would give 0.01, no floor 1.0, a floor at mean|r| 0.0388)
    ref = np.array([10.0, 0.1, 0.1, 0.1])
    got = np.array([10.0, 0.1, 0.1, 0.2])
    want = 0.1 / math.sqrt(25.0075)
    assert M.floored_rel_err(got, ref) == pytest.approx(want, rel=1e-12)


def test_large_entries_use_their_own_magnitude():
    # |r| above the rms: the denominator is |r| itself; the sign of the difference
    # does not matter
    ref = np.array([0.0, 0.0, 0.0, 8.0])          # rms = 4
    got = np.array([0.0, 0.0, 0.0, 7.2])
    assert M.floored_rel_err(got, ref) == pytest.approx(0.8 / 8.0, rel=1e-12)
    got2 = np.array([0.0, 0.0, 0.0, 8.8])
    assert M.floored_rel_err(got2, ref) == pytest.approx(0.8 / 8.0, rel=1e-12)
    # a negative reference entry: |r| = 8
    assert M.floored_rel_err(-got, -ref) == pytest.approx(0.1, rel=1e-12)


def test_explicit_floor():
    ref = np.array([1e-3, 2e-3])
    got = np.array([2e-3, 2e-3])
    assert M.floored_rel_err(got, ref, floor=0.5) == pytest.approx(1e-3 / 0.5, rel=1e-12)


def test_non_finite_results_fail():
    ref = np.array([1.0, 2.0, 3.0])
    assert M.floored_rel_err(np.array([1.0, np.nan, 3.0]), ref) == math.inf
    assert M.floored_rel_err(np.array([1.0, np.inf, 3.0]), ref) == math.inf
    assert not M.floored_rel_err(np.array([np.nan, 2.0, 3.0]), ref) <= 1.0


def test_all_zero_reference_and_empty():
    # rms 0: the denominators fall back to 1 (an absolute error)
    assert M.floored_rel_err(np.array([0.0, 1e-3]), np.zeros(2)) == pytest.approx(1e-3, rel=1e-12)
    assert M.floored_rel_err(np.zeros(0), np.zeros(0)) == 0.0


def test_identical_tensors_and_shape_check():
    r = np.random.default_rng(0).standard_normal(64)
    assert M.floored_rel_err(r.copy(), r) == 0.0
    with pytest.raises(AssertionError):
        M.floored_rel_err(np.zeros(3), np.zeros(4))


def test_report_fields_by_hand():
    ref = np.array([2.0, 0.0, -1.0, 1.0])          # rms = sqrt(6 / 4)
    got = np.array([2.5, 0.1, -1.0, 0.9])
    rep = M.report(got, ref)
    rms = math.sqrt(1.5)
    assert rep["err"] == pytest.approx(max(0.5 / 2.0, 0.1 / rms, 0.1 / rms), rel=1e-12)
    assert rep["max_abs"] == pytest.approx(0.5, rel=1e-12)
    # the unfloored ratio skips the zero reference entry: max(0.25, 0, 0.1)
    assert rep["max_rel_unfloored"] == pytest.approx(0.25, rel=1e-12)
    assert rep["rms_ref"] == pytest.approx(rms, rel=1e-12)


def test_tolerances_are_the_stated_bars():
    assert M.TOL == {"f32": 1e-5, "bf16": 2e-2}
