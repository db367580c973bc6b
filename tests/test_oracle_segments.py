"""Pins of the fp64 segment composition (oracle/segments.py): split runs
equal the serial run, a carry applied to any start state equals the
recurrence from it, closed forms, and planted mistakes that the pins catch."""

import math

import numpy as np
import pytest

from oracle import recurrence, segments


@pytest.fixture(scope="module")
def lib():
    return recurrence.OracleLib(recurrence.build_oracle())


def _head(T, K, V, seed, g_low=-0.5, beta_max=1.0):
    r = np.random.default_rng(seed)
    q = r.standard_normal((T, K))
    k = r.standard_normal((T, K))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = r.standard_normal((T, V))
    g = r.uniform(g_low, 0.0, T)
    beta = r.uniform(0.0, beta_max, T)
    S0 = r.standard_normal((K, V))
    return q, k, v, g, beta, S0


def _rel(x, r):
    return float(np.max(np.abs(x - r)) / max(np.max(np.abs(r)), 1e-300))


@pytest.mark.parametrize("T,cuts", [(17, [8]), (64, [1, 2, 63]), (200, [50, 100, 150]),
                                    (129, [64]), (96, list(range(6, 96, 6))), (40, [39])])
def test_segmented_equals_serial(lib, T, cuts):
    """Carries composed across 1 to 16 cut points (segments of one token
    included) reproduce the serial run's outputs and final state."""
    q, k, v, g, beta, S0 = _head(T, 6, 5, seed=T + len(cuts), beta_max=2.0)
    o_ref, S_ref = lib.fwd_head(q, k, v, g, beta, 0.45, S0)
    o, S, _ = segments.segmented_fwd(lib.fwd_head, q, k, v, g, beta, 0.45, S0, cuts)
    assert _rel(o, o_ref) < 1e-12, _rel(o, o_ref)
    assert _rel(S, S_ref) < 1e-12, _rel(S, S_ref)


def test_slow_decay_many_segments(lib):
    """cuLA issue #126's regime: decay close to 1 (g = -1e-3), many segments;
    in fp64 the composition stays exact."""
    q, k, v, g, beta, S0 = _head(512, 8, 4, seed=5)
    g[:] = -1e-3
    beta = 1.0 / (1.0 + np.exp(-(np.random.default_rng(6).standard_normal(512) - 2.0)))
    o_ref, S_ref = lib.fwd_head(q, k, v, g, beta, 0.35, S0)
    for nseg in (2, 4, 8, 16):
        cuts = [512 * i // nseg for i in range(1, nseg)]
        o, S, _ = segments.segmented_fwd(lib.fwd_head, q, k, v, g, beta, 0.35, S0, cuts)
        assert _rel(o, o_ref) < 1e-12 and _rel(S, S_ref) < 1e-12, nseg


def test_carry_is_the_segment_map(lib):
    """M S + b equals the recurrence's end state from any start state S."""
    q, k, v, g, beta, _ = _head(37, 5, 4, seed=9, beta_max=2.0)
    M, b = segments.segment_carry(k, v, g, beta)
    for seed in range(3):
        S = np.random.default_rng(seed).standard_normal((5, 4))
        _, S_end = lib.fwd_head(q, k, v, g, beta, 1.0, S)
        assert _rel(M @ S + b, S_end) < 1e-12


def test_closed_forms():
    """beta = 0: the carry is pure decay, M = exp(sum g) I and b = 0; one token
    with beta = 1 and a unit key: M = alpha (I - k k^T), b = k v^T."""
    q, k, v, g, beta, _ = _head(9, 4, 3, seed=3)
    M, b = segments.segment_carry(k, v, g, np.zeros(9))
    assert np.allclose(M, math.exp(g.sum()) * np.eye(4), rtol=1e-14, atol=1e-15)
    assert np.array_equal(b, np.zeros((4, 3)))
    M, b = segments.segment_carry(k[:1], v[:1], g[:1], np.ones(1))
    assert np.allclose(M, math.exp(g[0]) * (np.eye(4) - np.outer(k[0], k[0])), rtol=1e-14, atol=1e-15)
    assert np.allclose(b, np.outer(k[0], v[0]), rtol=1e-14, atol=1e-15)


def test_planted_mistakes_are_caught(lib):
    """Composing in the wrong order, dropping the decay from the carry, or
    transposing the transition each break the serial-equality pin."""
    q, k, v, g, beta, S0 = _head(60, 5, 4, seed=21, beta_max=2.0)
    cuts = [20, 40]
    o_ref, S_ref = lib.fwd_head(q, k, v, g, beta, 0.5, S0)
    edges = [0] + cuts + [60]

    def carries(fn):
        return [fn(k[a:e], v[a:e], g[a:e], beta[a:e]) for a, e in zip(edges[:-1], edges[1:])]

    def no_decay(kk, vv, gg, bb):
        return segments.segment_carry(kk, vv, np.zeros_like(gg), bb)

    def transposed(kk, vv, gg, bb):
        M, b = segments.segment_carry(kk, vv, gg, bb)
        return M.T, b

    def reversed_order(cs, S):
        starts = [S]
        for M, b in cs:
            starts.append(M @ (starts[-1] + b))  # carry added before the transition
        return starts[:-1], starts[-1]

    for cs, comp in [(carries(no_decay), segments.compose), (carries(transposed), segments.compose),
                     (carries(segments.segment_carry), reversed_order)]:
        starts, S = comp(cs, S0)
        assert _rel(S, S_ref) > 1e-6


# ---------------------------------------------------------------------------
# the per-channel-gate (KDA) variant, the kernel cuLA issue #126 splits
# ---------------------------------------------------------------------------

def _head_kda(T, K, V, seed, g_low=-0.5, beta_max=1.0):
    q, k, v, _, beta, S0 = _head(T, K, V, seed, g_low, beta_max)
    g = np.random.default_rng(seed + 7).uniform(g_low, 0.0, (T, K))
    return q, k, v, g, beta, S0


@pytest.mark.parametrize("T,cuts", [(17, [8]), (64, [1, 2, 63]), (200, [50, 100, 150]), (96, list(range(6, 96, 6)))])
def test_kda_segmented_equals_serial(T, cuts):
    """Per-channel decays: carries composed across 1 to 15 cut points
    reproduce the serial token loop's outputs and final state."""
    from oracle import kda
    q, k, v, g, beta, S0 = _head_kda(T, 6, 5, seed=100 + T, beta_max=2.0)
    o_ref, S_ref = kda.kda_fwd_head(q, k, v, g, beta, 0.45, S0)
    o, S, _ = segments.segmented_fwd(kda.kda_fwd_head, q, k, v, g, beta, 0.45, S0, cuts)
    assert _rel(o, o_ref) < 1e-12 and _rel(S, S_ref) < 1e-12


def test_kda_slow_decay_many_segments():
    """#126's regime for its own kernel: per-channel decay close to 1
    (g = -1e-3 on every channel, with a spread), beta = sigmoid(N(0,1) - 2),
    2 to 16 segments; in fp64 the composition stays exact."""
    from oracle import kda
    q, k, v, _, _, S0 = _head(512, 8, 4, seed=105)
    g = -1e-3 * np.random.default_rng(106).uniform(0.5, 1.5, (512, 8))
    beta = 1.0 / (1.0 + np.exp(-(np.random.default_rng(107).standard_normal(512) - 2.0)))
    o_ref, S_ref = kda.kda_fwd_head(q, k, v, g, beta, 0.35, S0)
    for nseg in (2, 4, 8, 16):
        cuts = [512 * i // nseg for i in range(1, nseg)]
        o, S, _ = segments.segmented_fwd(kda.kda_fwd_head, q, k, v, g, beta, 0.35, S0, cuts)
        assert _rel(o, o_ref) < 1e-12 and _rel(S, S_ref) < 1e-12, nseg


def test_kda_carry_is_the_segment_map():
    """M S + b equals the per-channel recurrence's end state from any S."""
    from oracle import kda
    q, k, v, g, beta, _ = _head_kda(37, 5, 4, seed=108, beta_max=2.0)
    M, b = segments.segment_carry(k, v, g, beta)
    for seed in range(3):
        S = np.random.default_rng(seed).standard_normal((5, 4))
        _, S_end = kda.kda_fwd_head(q, k, v, g, beta, 1.0, S)
        assert _rel(M @ S + b, S_end) < 1e-12


def test_kda_carry_planted_mistake_is_caught():
    """Putting the per-channel decay on the left of the write
    (diag(exp g) (I - beta k k^T), i.e. decaying after the read) breaks the
    carry pin; with a scalar gate the two orders agree, so only the
    per-channel case can tell them apart."""
    from oracle import kda
    q, k, v, g, beta, _ = _head_kda(20, 5, 4, seed=109, beta_max=2.0)
    n, K = k.shape
    M = np.eye(K)
    b = np.zeros((K, 4))
    for t in range(n):
        A = np.exp(g[t])[:, None] * (np.eye(K) - beta[t] * np.outer(k[t], k[t]))
        M = A @ M
        b = A @ b + beta[t] * np.outer(k[t], v[t])
    S = np.random.default_rng(3).standard_normal((5, 4))
    _, S_end = kda.kda_fwd_head(q, k, v, g, beta, 1.0, S)
    assert _rel(M @ S + b, S_end) > 1e-6
