"""Pins of the fp64 per-channel-gate (KDA) oracle: equal channels reduce to
the scalar-gate C oracle, beta = 0 is pure per-channel decay, the T = 1
closed form, and planted mistakes that the pins catch."""

import numpy as np
import pytest

from oracle import kda, recurrence


@pytest.fixture(scope="module")
def lib():
    return recurrence.OracleLib(recurrence.build_oracle())


def _head(T, K, V, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, K))
    k = rng.standard_normal((T, K))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, V))
    g = -rng.uniform(0.0, 0.5, (T, K))
    beta = rng.uniform(0.0, 1.0, T)
    S0 = rng.standard_normal((K, V)) / np.sqrt(K)
    return q, k, v, g, beta, S0


def test_equal_channels_equal_the_scalar_gate(lib):
    q, k, v, g, beta, S0 = _head(37, 6, 5, 0)
    gs = g[:, 0]
    o1, S1 = kda.kda_fwd_head(q, k, v, np.repeat(gs[:, None], 6, axis=1), beta, 0.4, S0)
    o2, S2 = lib.fwd_head(q, k, v, gs, beta, 0.4, S0)
    assert np.max(np.abs(o1 - o2)) <= 1e-13 * max(1.0, np.max(np.abs(o2)))
    assert np.max(np.abs(S1 - S2)) <= 1e-13 * max(1.0, np.max(np.abs(S2)))


def test_beta_zero_is_pure_per_channel_decay():
    q, k, v, g, beta, S0 = _head(20, 4, 3, 1)
    o, S = kda.kda_fwd_head(q, k, v, g, np.zeros(20), 0.7, S0)
    G = np.cumsum(g, axis=0)
    assert np.allclose(S, np.exp(G[-1])[:, None] * S0, rtol=1e-14, atol=1e-15)
    for t in (0, 7, 19):
        ref = 0.7 * ((np.exp(G[t])[:, None] * S0).T @ q[t])
        assert np.allclose(o[t], ref, rtol=1e-13, atol=1e-14)


def test_t1_closed_form():
    q, k, v, g, beta, S0 = _head(1, 5, 4, 2)
    a = np.exp(g[0])
    S1 = a[:, None] * S0 + beta[0] * np.outer(k[0], v[0] - (a[:, None] * S0).T @ k[0])
    o, S = kda.kda_fwd_head(q, k, v, g, beta, 0.3, S0)
    assert np.allclose(S, S1, rtol=1e-14, atol=1e-15)
    assert np.allclose(o[0], 0.3 * S1.T @ q[0], rtol=1e-14, atol=1e-15)


def test_planted_mistakes_are_caught():
    """Decaying the value columns instead of the key rows, or reading the
    state before the decay, breaks a pin."""
    q, k, v, g, beta, S0 = _head(1, 4, 4, 3)
    a = np.exp(g[0])

    def columns(S):
        return S * a[None, :]

    # the T = 1 closed form distinguishes row from column decay
    S_wrong = columns(S0) + beta[0] * np.outer(k[0], v[0] - columns(S0).T @ k[0])
    _, S = kda.kda_fwd_head(q, k, v, g, beta, 1.0, S0)
    assert not np.allclose(S, S_wrong, rtol=1e-6)
    S_late = a[:, None] * (S0 + beta[0] * np.outer(k[0], v[0] - S0.T @ k[0]))
    assert not np.allclose(S, S_late, rtol=1e-6)
