"""fp64 segment composition of the gated delta rule -- TEST INFRASTRUCTURE ONLY.

Only tests/ use this module; the CUDA library shares no code with it and has
no segmented path.  It states the identity that splitting one sequence into
segments relies on: cuLA issue #126 ("Hypothesis") describes intracard context
parallelism as per-segment affine transforms of the state (m_seg, b_seg) whose
carries are composed in order, and asks for coverage with more than two
segments and slow decay.

Per token (the "Research Sprint Day 1" update, S is K x V):
    S <- alpha S;  S <- S + beta k (v - S^T k)^T
which is affine in the previous state,
    S_t = A_t S_{t-1} + B_t,   A_t = alpha_t (I - beta_t k_t k_t^T),   B_t = beta_t k_t v_t^T.
A segment of tokens t = 1 .. n therefore maps its start state to its end state
by S_end = M S_start + b with
    M = A_n ... A_1,   b = sum_t (A_n ... A_{t+1}) B_t,
computed here left to right (M <- A_t M, b <- A_t b + B_t), independently of
S_start.  The start state of segment j + 1 is the composition
    S_start(j + 1) = M_j S_start(j) + b_j,
and each segment then runs the ordinary recurrence from its true start.

#126's own kernel is the per-channel-gate (KDA) variant, where the decay is
diag(exp(g_t)) with g_t in R^K; there the per-token map is
    A_t = (I - beta_t k_t k_t^T) diag(exp(g_t)),   B_t = beta_t k_t v_t^T
(the decay scales the key rows before the read, so it sits on the right), and
the same carries and composition apply.  segment_carry takes g of shape (n,)
or (n, K) and builds the matching A_t.
"""

from __future__ import annotations

import numpy as np


def segment_carry(k, v, g, beta):
    """(M (K x K), b (K x V)) of one segment: k (n, K), v (n, V), beta (n,);
    g (n,) for one decay per token, or (n, K) for one per key channel."""
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(g, np.float64)
    beta = np.asarray(beta, np.float64)
    n, K = k.shape
    M = np.eye(K)
    b = np.zeros((K, v.shape[1]))
    for t in range(n):
        A = (np.eye(K) - beta[t] * np.outer(k[t], k[t])) * np.exp(g[t])   # columns scaled: (.) diag(exp g)
        M = A @ M
        b = A @ b + beta[t] * np.outer(k[t], v[t])
    return M, b


def compose(carries, S0):
    """Start states of every segment and the end state, from the segments'
    carries [(M_j, b_j)] in order and the sequence's initial state S0."""
    starts = [np.array(S0, dtype=np.float64)]
    for M, b in carries:
        starts.append(M @ starts[-1] + b)
    return starts[:-1], starts[-1]


def segmented_fwd(run_segment, q, k, v, g, beta, scale, S0, cuts):
    """One (sequence, head) split at token indices ``cuts`` (0 < c < T,
    increasing): carries of every segment (independent of each other), their
    composition, then every segment from its true start state through
    ``run_segment(q, k, v, g, beta, scale, S_start) -> (o, S_end)`` (the
    per-token recurrence).  Returns (o (T, V), S_final, start states)."""
    T, K = np.shape(k)
    V = np.shape(v)[1]
    S0 = np.zeros((K, V)) if S0 is None else np.asarray(S0, np.float64)
    edges = [0] + list(cuts) + [T]
    carries = [segment_carry(k[a:e], v[a:e], g[a:e], beta[a:e]) for a, e in zip(edges[:-1], edges[1:])]
    starts, S_final = compose(carries, S0)
    o = np.zeros((T, V))
    for (a, e), Ss in zip(zip(edges[:-1], edges[1:]), starts):
        o[a:e], _ = run_segment(q[a:e], k[a:e], v[a:e], g[a:e], beta[a:e], scale, Ss)
    return o, S_final, starts
