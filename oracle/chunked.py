"""fp64 chunked (WY / UT-transform) algebra of the gated delta rule --
TEST INFRASTRUCTURE ONLY.

A second, independent formulation of the same operator, written with numpy
matrix products in fp64.  In exact arithmetic it reaches the per-token
recurrence's result exactly; the tests pin the two against each other to
~1e-12, which checks both.  It also spells out, step by step, the chunk
intermediates that the fla issue #1550 "Intermediate rounding diagnosis"
names (triangular inverse, causal QK score matrix, write product, WY value
tensor u), and the reverse-mode algebra through them.

Notation, per chunk of n <= C tokens with chunk-start state S0 (K x V):
  G_i   = sum_{j<=i} g_j                     (log decay kept as a cumsum of g,
                                              "Research Sprint Day 2", step 5)
  gam_i = exp(G_i),  gam_C = exp(G_n)
  A_ij  = beta_i (k_i . k_j) exp(G_i - G_j)  for j < i, else 0
  Tm    = (I + A)^-1                          (unit lower triangular)
  w     = Tm diag(beta gam) K,   u = Tm diag(beta) V
  Delta = u - w S0                            (= beta_i e_i of the recurrence)
  O     = scale [diag(gam) Q S0 + (Q K^T o M) Delta],
          M_ij = exp(G_i - G_j) for j <= i (diagonal included), else 0
  S1    = gam_C S0 + K^T diag(exp(G_n - G_j)) Delta
Exponents are masked BEFORE exp (only i >= j pairs are exponentiated), so
every exponent is <= 0.
"""

from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


def _decay_matrix(G, include_diag):
    n = G.shape[0]
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    mask = (i >= j) if include_diag else (i > j)
    expo = np.where(mask, G[:, None] - G[None, :], -np.inf)
    return np.exp(expo)


def _chunk_forward(Q, K, V, g, beta, S0):
    n = Q.shape[0]
    G = np.cumsum(g)
    gam = np.exp(G)
    Ms = _decay_matrix(G, include_diag=False)
    M = _decay_matrix(G, include_diag=True)
    KK = K @ K.T
    A = beta[:, None] * KK * Ms
    Tm = solve_triangular(np.eye(n) + A, np.eye(n), lower=True, unit_diagonal=True)
    w = Tm @ ((beta * gam)[:, None] * K)
    u = Tm @ (beta[:, None] * V)
    Delta = u - w @ S0
    QK = Q @ K.T
    P = QK * M
    dec = np.exp(G[-1] - G)
    return dict(G=G, gam=gam, Ms=Ms, M=M, KK=KK, A=A, Tm=Tm, w=w, u=u, Delta=Delta,
                QK=QK, P=P, dec=dec)


def fwd_head(q, k, v, g, beta, scale, S0=None, chunk=64):
    """Chunked forward for one (sequence, head).  Returns (o, S_final, chunks)
    where chunks is the list of per-chunk intermediates (for diagnosis)."""
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    T, K = q.shape
    V = v.shape[1]
    S = np.zeros((K, V)) if S0 is None else np.array(S0, dtype=np.float64)
    o = np.zeros((T, V))
    inter = []
    for c0 in range(0, T, chunk):
        c1 = min(c0 + chunk, T)
        Q, Kc, Vc, gc, bc = q[c0:c1], k[c0:c1], v[c0:c1], g[c0:c1], beta[c0:c1]
        f = _chunk_forward(Q, Kc, Vc, gc, bc, S)
        o[c0:c1] = scale * (f["gam"][:, None] * (Q @ S) + f["P"] @ f["Delta"])
        f["S0"] = S
        S = f["gam"][-1] * S + (Kc * f["dec"][:, None]).T @ f["Delta"]
        inter.append(f)
    return o, S, inter


def bwd_head(q, k, v, g, beta, scale, S0, dO, dS_final, chunk=64):
    """Reverse mode of the chunked algebra for one (sequence, head).

    Walks chunks from last to first carrying dS (gradient w.r.t. the chunk-end
    state).  Returns dict of dq, dk, dv, dg, dbeta, dS0 (fp64)."""
    q, k, v, g, beta, dO = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta, dO))
    T, K = q.shape
    V = v.shape[1]
    _, _, inter = fwd_head(q, k, v, g, beta, scale, S0, chunk)
    dS = np.zeros((K, V)) if dS_final is None else np.array(dS_final, dtype=np.float64)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dg = np.zeros_like(g)
    dbeta = np.zeros_like(beta)
    starts = list(range(0, T, chunk))
    for ci in range(len(starts) - 1, -1, -1):
        c0 = starts[ci]
        c1 = min(c0 + chunk, T)
        f = inter[ci]
        Q, Kc, Vc, bc = q[c0:c1], k[c0:c1], v[c0:c1], beta[c0:c1]
        dOc = dO[c0:c1]
        S0c = f["S0"]
        gam, dec, Delta, Tm = f["gam"], f["dec"], f["Delta"], f["Tm"]
        n = c1 - c0
        dQ = np.zeros((n, K))
        dK = np.zeros((n, K))
        dG = np.zeros(n)
        dgam = np.zeros(n)
        dbc = np.zeros(n)
        # output: O = scale [diag(gam) Q S0 + P Delta]
        QS = Q @ S0c
        dQS = scale * gam[:, None] * dOc
        dQ += dQS @ S0c.T
        dS0 = Q.T @ dQS
        dgam += scale * np.sum(QS * dOc, axis=1)
        dP = scale * dOc @ Delta.T
        dDelta = scale * f["P"].T @ dOc
        dQK = dP * f["M"]
        dQ += dQK @ Kc
        dK += dQK.T @ Q
        dMw = dP * f["QK"] * f["M"]
        dG += dMw.sum(axis=1) - dMw.sum(axis=0)
        # state: S1 = gam_C S0 + K^T diag(dec) Delta
        dS0 += gam[-1] * dS
        dgam[-1] += np.sum(dS * S0c)
        KdS = Kc @ dS
        dK += (dec[:, None] * Delta) @ dS.T
        dDelta += dec[:, None] * KdS
        ddec = np.sum(KdS * Delta, axis=1) * dec
        dG[-1] += ddec.sum()
        dG -= ddec
        # Delta = Tm Bhat, Bhat = diag(beta) V - diag(beta gam) K S0
        dBhat = Tm.T @ dDelta
        dA = -(dBhat @ Delta.T) * (f["Ms"] > 0)
        KS = Kc @ S0c
        dv[c0:c1] = bc[:, None] * dBhat
        rowVB = np.sum(Vc * dBhat, axis=1)
        rowKSB = np.sum(KS * dBhat, axis=1)
        dbc += rowVB - gam * rowKSB
        dgam += -bc * rowKSB
        dKS = -(bc * gam)[:, None] * dBhat
        dK += dKS @ S0c.T
        dS0 += Kc.T @ dKS
        # A = diag(beta) (K K^T o Ms)
        KKM = f["KK"] * f["Ms"]
        dbc += np.sum(dA * KKM, axis=1)
        dKK = dA * bc[:, None] * f["Ms"]
        dK += dKK @ Kc + dKK.T @ Kc
        dMs = dA * bc[:, None] * f["KK"] * f["Ms"]
        dG += dMs.sum(axis=1) - dMs.sum(axis=0)
        # gam = exp(G); G = cumsum(g)
        dG += dgam * gam
        dg[c0:c1] = np.cumsum(dG[::-1])[::-1]
        dq[c0:c1] = dQ
        dk[c0:c1] = dK
        dbeta[c0:c1] = dbc
        dS = dS0
    return dict(dq=dq, dk=dk, dv=dv, dg=dg, dbeta=dbeta, dS0=dS)
