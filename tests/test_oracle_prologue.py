"""Pins of the fp64 prologue oracle (q/k L2 normalisation, gates, their
reverse mode): closed forms, invariants, central finite differences, and
planted mistakes that the pins must catch."""

import math

import numpy as np
import pytest

from oracle import prologue as P


def test_closed_forms():
    assert P.softplus(0.0) == pytest.approx(math.log(2.0), abs=1e-15)
    assert P.sigmoid(0.0) == pytest.approx(0.5, abs=1e-15)
    # large arguments: softplus(x) -> x, sigmoid stays finite
    assert P.softplus(50.0) == pytest.approx(50.0, rel=1e-15)
    assert P.sigmoid(-800.0) == pytest.approx(0.0, abs=1e-300)
    y = P.l2norm(np.array([3.0, 4.0]))
    assert np.allclose(y, np.array([3.0, 4.0]) / math.sqrt(25.0 + P.EPS), rtol=0, atol=1e-15)
    assert np.array_equal(P.l2norm(np.zeros((2, 8))), np.zeros((2, 8)))
    # decay gate at u = 0, A_log = 0: g = -ln 2; bounded gate at u = 0: lower / 2
    g, beta = P.gates(np.zeros((1, 1)), np.zeros((1, 1)), A_log=np.zeros(1), mode="decay")
    assert g[0, 0] == pytest.approx(-math.log(2.0), abs=1e-15) and beta[0, 0] == 0.5
    g, beta = P.gates(np.zeros((1, 1)), np.zeros((1, 1)), mode="bounded", lower=-5.0, beta_scale=2.0)
    assert g[0, 0] == pytest.approx(-2.5, abs=1e-15) and beta[0, 0] == 1.0


def test_ranges_and_unit_norm():
    rng = np.random.default_rng(0)
    a = rng.standard_normal((64, 5)) * 4
    b = rng.standard_normal((64, 5)) * 4
    A_log = rng.uniform(0, math.log(16), 5)
    dtb = rng.uniform(-1, 1, 5)
    g, beta = P.gates(a, b, A_log, dtb, mode="decay")
    assert np.all(g <= 0) and np.all((beta > 0) & (beta < 1))
    g, beta = P.gates(a, b, None, dtb, mode="bounded", lower=-5.0, beta_scale=2.0)
    assert np.all((g > -5.0) & (g < 0)) and np.all((beta > 0) & (beta < 2))
    x = rng.standard_normal((32, 128))
    assert np.allclose(np.linalg.norm(P.l2norm(x), axis=-1), 1.0, atol=1e-7)


def _fd_check(f, args, grads, eps=1e-6, rtol=1e-7):
    """Central differences of the scalar f(*args) against the given gradients."""
    for idx, (arg, grad) in enumerate(zip(args, grads)):
        if grad is None:
            continue
        num = np.zeros_like(arg)
        it = np.nditer(arg, flags=["multi_index"])
        for _ in it:
            mi = it.multi_index
            a1 = [x.copy() for x in args]
            a2 = [x.copy() for x in args]
            a1[idx][mi] += eps
            a2[idx][mi] -= eps
            num[mi] = (f(*a1) - f(*a2)) / (2 * eps)
        err = np.max(np.abs(num - grad)) / max(np.max(np.abs(num)), 1e-30)
        assert err < rtol, (idx, err)


def test_l2norm_reverse_mode_finite_differences():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 6))
    w = rng.standard_normal((3, 6))
    f = lambda x_: float(np.sum(w * P.l2norm(x_)))  # noqa: E731
    _fd_check(f, [x], [P.l2norm_bwd(x, w)])


@pytest.mark.parametrize("mode,beta_scale", [("decay", 1.0), ("decay", 2.0), ("bounded", 1.0)])
def test_gates_reverse_mode_finite_differences(mode, beta_scale):
    rng = np.random.default_rng(2)
    T, H = 4, 3
    a = rng.standard_normal((T, H))
    b = rng.standard_normal((T, H))
    A_log = rng.uniform(0, math.log(16), H)
    dtb = rng.uniform(-1, 1, H)
    wg = rng.standard_normal((T, H))
    wb = rng.standard_normal((T, H))

    def f(a_, b_, A_, d_):
        g, beta = P.gates(a_, b_, A_ if mode == "decay" else None, d_, mode=mode, lower=-5.0,
                          beta_scale=beta_scale)
        return float(np.sum(wg * g) + np.sum(wb * beta))

    da, db, dA, dd = P.gates_bwd(a, b, wg, wb, A_log if mode == "decay" else None, dtb, mode=mode,
                                 lower=-5.0, beta_scale=beta_scale)
    _fd_check(f, [a, b, A_log, dtb], [da, db, dA, dd])


def test_planted_mistakes_are_caught():
    """Plausible slips in the reverse mode fail the finite-difference pin."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 5))
    w = rng.standard_normal((2, 5))
    f = lambda x_: float(np.sum(w * P.l2norm(x_)))  # noqa: E731

    def no_projection(x_, dy):
        r = 1.0 / np.sqrt(np.sum(x_ * x_, axis=-1, keepdims=True) + P.EPS)
        return r * dy

    def wrong_sign(x_, dy):
        r = 1.0 / np.sqrt(np.sum(x_ * x_, axis=-1, keepdims=True) + P.EPS)
        y = x_ * r
        return r * (dy + y * np.sum(y * dy, axis=-1, keepdims=True))

    for bad in (no_projection, wrong_sign):
        with pytest.raises(AssertionError):
            _fd_check(f, [x], [bad(x, w)])
    # the decay gate's A_log gradient with g replaced by softplus (dropped -exp(A_log))
    a = rng.standard_normal((3, 2))
    b = rng.standard_normal((3, 2))
    A_log = rng.uniform(0, 2, 2)
    wg = rng.standard_normal((3, 2))

    def f2(A_):
        return float(np.sum(wg * P.gates(a, b, A_, None, mode="decay")[0]))

    with pytest.raises(AssertionError):
        _fd_check(f2, [A_log], [np.sum(wg * P.softplus(a), axis=0)])
