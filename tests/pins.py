"""Pins of the fp64 oracle: facts fixed by the pages and by mathematics.

Each pin takes a loaded oracle library (``oracle.recurrence.OracleLib``) so
that the same checks can be run against deliberately broken copies of the
oracle (see test_oracle_mutations.py).  A pin raises AssertionError when the
oracle disagrees with the fact it encodes.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

from oracle import chunked

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rand_head(T, K, V, seed, s0=True, beta_max=1.0, g_low=-0.5):
    r = np.random.default_rng(seed)
    q = r.standard_normal((T, K))
    k = r.standard_normal((T, K))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = r.standard_normal((T, V))
    g = r.uniform(g_low, 0.0, T)
    b = r.uniform(0.0, beta_max, T)
    S0 = r.standard_normal((K, V)) if s0 else None
    return q, k, v, g, b, S0


def _rel(x, r):
    return float(np.max(np.abs(np.asarray(x) - np.asarray(r))) / max(np.max(np.abs(r)), 1e-300))


def pin_page1_equals_page4(lib):
    """The page-1 loop (S is K x V) and the page-4 matrix form (S is V x K)
    are transposes of each other and give the same output."""
    for (T, K, V, seed) in [(40, 5, 3, 1), (33, 4, 7, 2), (70, 8, 8, 3)]:
        q, k, v, g, b, S0 = _rand_head(T, K, V, seed, beta_max=2.0)
        o1, S1 = lib.fwd_head(q, k, v, g, b, 0.37, S0)
        o2, R2 = lib.fwd_head_matrix_form(q, k, v, g, b, 0.37, S0.T.copy())
        assert _rel(o1, o2) < 1e-13, _rel(o1, o2)
        assert _rel(S1, R2.T) < 1e-13, _rel(S1, R2.T)


def pin_t1_closed_form(lib):
    """One token: S1 = alpha S0 + beta k (v - alpha S0^T k)^T, o = scale S1^T q;
    from S0 = 0 this is S1 = beta k v^T and o = scale beta (q.k) v."""
    q, k, v, g, b, S0 = _rand_head(1, 6, 5, 11)
    o, S = lib.fwd_head(q, k, v, g, b, 0.5, None)
    S_ref = b[0] * np.outer(k[0], v[0])
    o_ref = 0.5 * b[0] * np.dot(q[0], k[0]) * v[0]
    assert _rel(S, S_ref) < 1e-14 and _rel(o[0], o_ref) < 1e-14
    o, S = lib.fwd_head(q, k, v, g, b, 0.5, S0)
    a = math.exp(g[0])
    S_ref = a * S0 + b[0] * np.outer(k[0], v[0] - a * S0.T @ k[0])
    assert _rel(S, S_ref) < 1e-14
    assert _rel(o[0], 0.5 * S_ref.T @ q[0]) < 1e-14


def pin_t2_closed_form(lib):
    """Two tokens from S0 = 0:
    o2 = scale [a2 b1 (q2.k1 - b2 (q2.k2)(k2.k1)) v1 + b2 (q2.k2) v2]."""
    for seed in (5, 6):
        q, k, v, g, b, _ = _rand_head(2, 4, 3, seed, beta_max=2.0)
        o, _ = lib.fwd_head(q, k, v, g, b, 0.8, None)
        a2 = math.exp(g[1])
        ref = 0.8 * (a2 * b[0] * (q[1] @ k[0] - b[1] * (q[1] @ k[1]) * (k[1] @ k[0])) * v[0]
                     + b[1] * (q[1] @ k[1]) * v[1])
        assert _rel(o[1], ref) < 1e-14, _rel(o[1], ref)


def pin_golden_worked_example(lib):
    """Hand-derived two-token example (tests/golden/t2_worked_example.json)."""
    with open(os.path.join(GOLDEN, "t2_worked_example.json")) as f:
        ex = json.load(f)
    arr = lambda n: np.array(ex[n], dtype=np.float64)  # noqa: E731
    o, S = lib.fwd_head(arr("q"), arr("k"), arr("v"), arr("g"), arr("beta"), ex["scale"], None)
    assert np.max(np.abs(o - arr("o"))) < 1e-12
    assert np.max(np.abs(S - arr("S_final"))) < 1e-12


def pin_beta_zero_is_pure_decay(lib):
    """beta = 0: nothing is written, so S_T = exp(sum g) S0 and
    o_t = scale exp(G_t) S0^T q_t."""
    q, k, v, g, b, S0 = _rand_head(50, 6, 4, 21, g_low=-0.2)
    b = np.zeros_like(b)
    o, S = lib.fwd_head(q, k, v, g, b, 0.3, S0)
    G = np.cumsum(g)
    assert _rel(S, math.exp(G[-1]) * S0) < 1e-13
    o_ref = 0.3 * np.exp(G)[:, None] * (q @ S0)
    assert _rel(o, o_ref) < 1e-13


def pin_exact_recall_and_overwrite(lib):
    """alpha = 1, beta = 1, orthonormal keys: S = sum_j k_j v_j^T and querying
    with k_j returns v_j.  Writing k_j again with beta = 1 replaces v_j (the
    delta rule writes the error, not the value)."""
    K, V, n = 8, 5, 6
    r = np.random.default_rng(31)
    basis, _ = np.linalg.qr(r.standard_normal((K, K)))
    keys = basis[:, :n].T
    vals = r.standard_normal((n, V))
    # store n pairs, then query each key with beta = 0 (read-only tokens)
    k = np.concatenate([keys, keys])
    v = np.concatenate([vals, np.zeros((n, V))])
    q = np.concatenate([np.zeros((n, K)), keys])
    b = np.concatenate([np.ones(n), np.zeros(n)])
    g = np.zeros(2 * n)
    o, S = lib.fwd_head(q, k, v, g, b, 1.0, None)
    assert _rel(S, keys.T @ vals) < 1e-13
    assert _rel(o[n:], vals) < 1e-13
    # overwrite key 2 with a new value, then read it back
    new = r.standard_normal(V)
    k2 = np.concatenate([k[:n], keys[2:3], keys[2:3]])
    v2 = np.concatenate([v[:n], new[None], np.zeros((1, V))])
    q2 = np.concatenate([q[:n], np.zeros((1, K)), keys[2:3]])
    b2 = np.concatenate([b[:n], [1.0], [0.0]])
    o2, _ = lib.fwd_head(q2, k2, v2, np.zeros(n + 2), b2, 1.0, None)
    assert _rel(o2[-1], new) < 1e-13


def pin_linearity(lib):
    """From S0 = 0 the output is linear in v and in scale."""
    q, k, v, g, b, _ = _rand_head(30, 5, 4, 41)
    v2 = np.random.default_rng(42).standard_normal(v.shape)
    o1, _ = lib.fwd_head(q, k, v, g, b, 1.0, None)
    o2, _ = lib.fwd_head(q, k, v2, g, b, 1.0, None)
    o3, _ = lib.fwd_head(q, k, 2.0 * v - 3.0 * v2, g, b, 1.0, None)
    assert _rel(o3, 2.0 * o1 - 3.0 * o2) < 1e-12
    o4, _ = lib.fwd_head(q, k, v, g, b, 0.25, None)
    assert _rel(o4, 0.25 * o1) < 1e-14


def pin_chunked_algebra_agrees(lib):
    """The chunked WY algebra (an independent formulation) reaches the same
    result as the per-token loop, for several chunk sizes, partial last
    chunks and a strong decay (G far below the fp32 exp range)."""
    cases = [(150, 8, 6, 51, -0.5), (300, 16, 16, 52, -0.5), (65, 4, 4, 53, -5.0),
             (129, 8, 4, 54, -12.0)]
    for (T, K, V, seed, g_low) in cases:
        q, k, v, g, b, S0 = _rand_head(T, K, V, seed, beta_max=2.0, g_low=g_low)
        o1, S1 = lib.fwd_head(q, k, v, g, b, 0.4, S0)
        for C in (1, 7, 16, 64):
            o2, S2, _ = chunked.fwd_head(q, k, v, g, b, 0.4, S0, chunk=C)
            assert np.all(np.isfinite(o2))
            assert _rel(o2, o1) < 1e-12, (T, C, _rel(o2, o1))
            assert _rel(S2, S1) < 1e-12, (T, C, _rel(S2, S1))


def pin_finite_differences(lib):
    """Central finite differences of L = <o, dO> + <S_T, dS_T> in fp64 agree
    with the reverse mode for every input, on tiny sizes."""
    T, K, V = 7, 3, 4
    q, k, v, g, b, S0 = _rand_head(T, K, V, 61, beta_max=2.0)
    r = np.random.default_rng(62)
    dO = r.standard_normal((T, V))
    dSf = r.standard_normal((K, V))
    scale = 0.7

    def loss(args):
        o, S = lib.fwd_head(*args[:5], scale, args[5])
        return float(np.sum(o * dO) + np.sum(S * dSf))

    grads = lib.bwd_head(q, k, v, g, b, scale, S0, dO, dSf)
    args = [q, k, v, g, b, S0]
    names = ["dq", "dk", "dv", "dg", "dbeta", "dS0"]
    h = 1e-6
    for ai, name in enumerate(names):
        fd = np.zeros_like(args[ai])
        for idx in np.ndindex(args[ai].shape):
            ap = [a.copy() for a in args]
            am = [a.copy() for a in args]
            ap[ai][idx] += h
            am[ai][idx] -= h
            fd[idx] = (loss(ap) - loss(am)) / (2 * h)
        assert _rel(grads[name], fd) < 1e-7, (name, _rel(grads[name], fd))


def pin_chunked_reverse_mode_agrees(lib):
    """The reverse mode of the chunked algebra (derived independently of the
    per-token reverse mode) gives the same gradients."""
    for (T, K, V, seed, C) in [(150, 8, 6, 71, 64), (97, 4, 8, 72, 16), (20, 5, 3, 73, 7)]:
        q, k, v, g, b, S0 = _rand_head(T, K, V, seed, beta_max=2.0)
        r = np.random.default_rng(seed + 100)
        dO = r.standard_normal((T, V))
        dSf = r.standard_normal((K, V))
        g1 = lib.bwd_head(q, k, v, g, b, 0.6, S0, dO, dSf)
        g2 = chunked.bwd_head(q, k, v, g, b, 0.6, S0, dO, dSf, chunk=C)
        for name in g1:
            assert _rel(g2[name], g1[name]) < 1e-11, (name, _rel(g2[name], g1[name]))


ALL_PINS = [
    pin_page1_equals_page4,
    pin_t1_closed_form,
    pin_t2_closed_form,
    pin_golden_worked_example,
    pin_beta_zero_is_pure_decay,
    pin_exact_recall_and_overwrite,
    pin_linearity,
    pin_chunked_algebra_agrees,
    pin_finite_differences,
    pin_chunked_reverse_mode_agrees,
]
