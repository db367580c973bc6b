"""fp64 per-channel-gate (KDA) variant of the gated delta rule, token by
token -- TEST INFRASTRUCTURE ONLY.

Only tests/ use this module; the CUDA library shares no code with it.

cuLA issue #126 runs the KDA kernel (flash_kda_fwd) with a gate g of shape
(B, T, H, D): one log decay per key channel instead of one per head.  The
state update of the "Research Sprint Day 1" loop then decays each key row of
S by its own factor:
    S <- diag(exp(g_t)) S;  v_old = S^T k_t;  S <- S + beta_t k_t (v_t - v_old)^T;
    o_t = scale S^T q_t
(S is K x V, key rows i, value columns j).  With all channels equal it is the
scalar-gate operator, which a test pins against the C oracle.
"""

from __future__ import annotations

import numpy as np


def kda_fwd_head(q, k, v, g, beta, scale, S0=None):
    """One (sequence, head): q, k (T, K), v (T, V), g (T, K), beta (T,).
    Returns (o (T, V), S (K, V)) in fp64."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(g, np.float64)
    beta = np.asarray(beta, np.float64)
    T, K = k.shape
    V = v.shape[1]
    S = np.zeros((K, V)) if S0 is None else np.array(S0, dtype=np.float64)
    o = np.zeros((T, V))
    for t in range(T):
        S = np.exp(g[t])[:, None] * S          # forget, per key row
        v_old = S.T @ k[t]                     # read what is stored for k_t
        S = S + beta[t] * np.outer(k[t], v[t] - v_old)   # write the error
        o[t] = scale * (S.T @ q[t])
    return o, S


def kda_fwd(q, k, v, g, beta, scale, initial_state=None, cu_seqlens=None):
    """Batched: q, k (B, T, H, K), v (B, T, H, V), g (B, T, H, K), beta (B, T, H);
    packed sequences when cu_seqlens is given (B = 1).  Returns (o, S) with S of
    shape (N, H, K, V)."""
    B, T, H, K = np.shape(k)
    V = np.shape(v)[3]
    if cu_seqlens is None:
        bounds = [(b, 0, T) for b in range(B)]
    else:
        cu = np.asarray(cu_seqlens)
        bounds = [(0, int(cu[n]), int(cu[n + 1])) for n in range(len(cu) - 1)]
    o = np.zeros((B, T, H, V))
    S = np.zeros((len(bounds), H, K, V))
    for n, (b, t0, t1) in enumerate(bounds):
        for h in range(H):
            s0 = None if initial_state is None else initial_state[n, h]
            o_h, S_h = kda_fwd_head(q[b, t0:t1, h], k[b, t0:t1, h], v[b, t0:t1, h], g[b, t0:t1, h],
                                    beta[b, t0:t1, h], scale, s0)
            o[b, t0:t1, h] = o_h
            S[n, h] = S_h
    return o, S
