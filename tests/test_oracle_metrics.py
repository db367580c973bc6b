"""The error metrics every parity check goes through, pinned to values
worked out by hand (CPU only).

* rel_l2 is the relative L2 of the cuLA issue #126 reproduction (a 1e-30
  clamp on the reference norm) and the "relative RMS" output error of fla
  issue #1550: the norm of the difference divided by the norm of the
  REFERENCE, never of the result under test.
* max_rel is max|x - r| / max|r| over the whole tensor (the reading of
  "Research Sprint Day 1"'s max-relative error).
* window_rel_l2 splits the token axis into 8 windows of T // 8 tokens, the
  last one also taking the remainder (cuLA issue #126's per-window report).

Each check below is also run on planted mistakes (normalising by the wrong
tensor, no clamp, the remainder dropped, the wrong axis, an elementwise
max-relative), and every mistake must fail at least one check.
"""

import math
import types

import numpy as np
import pytest

from oracle import metrics


def _check_rel_l2(m):
    # x - r = (0, 2, 2): norm sqrt(8); |r| = 1; |x| = 3 (dividing by |x| gives 0.943)
    assert m.rel_l2([1.0, 2.0, 2.0], [1.0, 0.0, 0.0]) == pytest.approx(math.sqrt(8.0), rel=1e-15)
    # a 3-4-5 difference over a reference of norm 10
    assert m.rel_l2(np.array([[9.0, 4.0], [0.0, 0.0]]), np.array([[6.0, 0.0], [8.0, 0.0]])) == \
        pytest.approx(math.hypot(3.0, 4.0, 8.0) / 10.0, rel=1e-15)
    # the clamp: a zero reference divides by 1e-30
    assert m.rel_l2([3.0, 4.0], [0.0, 0.0]) == pytest.approx(5e30, rel=1e-12)
    assert m.rel_l2([0.0, 0.0], [0.0, 0.0]) == 0.0
    # exact agreement, and a uniform 1 % perturbation
    r = np.linspace(-2.0, 3.0, 17)
    assert m.rel_l2(r, r) == 0.0
    assert m.rel_l2(1.01 * r, r) == pytest.approx(0.01, rel=1e-12)


def _check_max_rel(m):
    # |x - r| = (1, 3, 2), max 3; max|r| = 8 -> 0.375 (elementwise would give 0.5,
    # dividing by max|x| = 5 would give 0.6)
    assert m.max_rel([1.0, 5.0, -2.0], [2.0, 8.0, -4.0]) == pytest.approx(0.375, rel=1e-15)
    # a sign flip of the largest entry doubles it
    assert m.max_rel([-4.0, 1.0], [4.0, 1.0]) == pytest.approx(2.0, rel=1e-15)
    # over the whole tensor, not per row: row 0's error against row 1's scale
    assert m.max_rel(np.array([[0.5, 0.0], [10.0, 0.0]]), np.array([[0.0, 0.0], [10.0, 0.0]])) == \
        pytest.approx(0.05, rel=1e-15)


def _check_windows(m):
    # T = 10 tokens, 8 windows of 1 token, the last one tokens 7..9
    r = np.ones(10)
    x = r + 0.1 * np.arange(10)
    expect = [0.1 * i for i in range(7)] + [math.sqrt((0.49 + 0.64 + 0.81) / 3.0)]
    got = m.window_rel_l2(x[None, :], r[None, :], axis=1)
    assert len(got) == 8
    assert got == pytest.approx(expect, rel=1e-12, abs=1e-15)
    # the same along axis 0 of a (T, H) array, two identical columns
    got0 = m.window_rel_l2(np.stack([x, x], 1), np.stack([r, r], 1), axis=0)
    assert got0 == pytest.approx(expect, rel=1e-12, abs=1e-15)
    # (B, T, H): the token axis is 1; a perturbation of one head in window 3 only
    rr = np.ones((2, 16, 3))
    xx = rr.copy()
    xx[:, 6:8, 1] += 3.0  # window 3 = tokens 6, 7 (T // 8 = 2)
    w = m.window_rel_l2(xx, rr, axis=1)
    assert w[3] == pytest.approx(math.sqrt(4 * 9.0) / math.sqrt(2 * 2 * 3), rel=1e-12)
    assert all(w[i] == 0.0 for i in range(8) if i != 3)


CHECKS = (_check_rel_l2, _check_max_rel, _check_windows)


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_metrics_pinned(check):
    check(metrics)


def _mutant(**overrides):
    ns = types.SimpleNamespace(rel_l2=metrics.rel_l2, max_rel=metrics.max_rel,
                               window_rel_l2=metrics.window_rel_l2)
    for k, f in overrides.items():
        setattr(ns, k, f)
    return ns


def _rel_by_result(x, r):
    x, r = np.asarray(x, float), np.asarray(r, float)
    return float(np.linalg.norm(x - r) / max(np.linalg.norm(x), 1e-30))


def _rel_no_clamp(x, r):
    x, r = np.asarray(x, float), np.asarray(r, float)
    with np.errstate(divide="ignore", invalid="ignore"):
        return float(np.linalg.norm(x - r) / np.linalg.norm(r))


def _rel_rms_mean(x, r):
    # RMS of the difference over RMS of ... the difference's length (not relative)
    x, r = np.asarray(x, float), np.asarray(r, float)
    return float(np.sqrt(np.mean((x - r) ** 2)))


def _max_elementwise(x, r):
    x, r = np.asarray(x, float), np.asarray(r, float)
    return float(np.max(np.abs(x - r) / np.maximum(np.abs(r), 1e-30)))


def _max_by_result(x, r):
    x, r = np.asarray(x, float), np.asarray(r, float)
    return float(np.max(np.abs(x - r)) / max(np.max(np.abs(x)), 1e-30))


def _max_per_row(x, r):
    x, r = np.atleast_2d(np.asarray(x, float)), np.atleast_2d(np.asarray(r, float))
    return float(np.max(np.max(np.abs(x - r), -1) / np.maximum(np.max(np.abs(r), -1), 1e-30)))


def _win_remainder_dropped(x, r, axis=1, windows=8):
    x, r = np.asarray(x, float), np.asarray(r, float)
    w = x.shape[axis] // windows
    out = []
    for i in range(windows):
        sl = [slice(None)] * x.ndim
        sl[axis] = slice(i * w, (i + 1) * w)
        out.append(metrics.rel_l2(x[tuple(sl)], r[tuple(sl)]))
    return out


def _win_wrong_axis(x, r, axis=1, windows=8):
    return metrics.window_rel_l2(x, r, axis=x.ndim - 1 if axis != x.ndim - 1 else 0, windows=windows)


def _win_pooled(x, r, axis=1, windows=8):
    # one norm over all windows instead of one per window
    return [metrics.rel_l2(x, r)] * windows


MUTANTS = [
    ("rel_l2 divides by the result's norm", dict(rel_l2=_rel_by_result)),
    ("rel_l2 without the 1e-30 clamp", dict(rel_l2=_rel_no_clamp)),
    ("rel_l2 is an absolute RMS", dict(rel_l2=_rel_rms_mean)),
    ("max_rel elementwise", dict(max_rel=_max_elementwise)),
    ("max_rel divides by the result", dict(max_rel=_max_by_result)),
    ("max_rel per row", dict(max_rel=_max_per_row)),
    ("windows drop the remainder", dict(window_rel_l2=_win_remainder_dropped)),
    ("windows on the wrong axis", dict(window_rel_l2=_win_wrong_axis)),
    ("windows pooled", dict(window_rel_l2=_win_pooled)),
]


def _fails_a_check(ns):
    for check in CHECKS:
        try:
            with np.errstate(all="ignore"):
                check(ns)
        except (AssertionError, ValueError, IndexError, ZeroDivisionError):
            return True
    return False


@pytest.mark.parametrize("name,overrides", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_metric_mistake_is_caught(name, overrides):
    assert _fails_a_check(_mutant(**overrides)), name
