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

kda_chunk_fwd_head is a second formulation of the same operator: the chunk
algebra with the per-channel decay inside the key dot products (the form a
chunked kernel evaluates).  In exact arithmetic it equals the token loop; the
tests pin the two against each other to ~1e-12.

kda_bwd_head is the reverse mode of the token loop (gradients of
L = <o, dO> + <S_T, dS_T> with respect to every input), pinned by central
finite differences and, with all channels equal, by the scalar-gate C
oracle's reverse mode.
"""

from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


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


def _kda_chunk(Q, Kc, Vc, gc, bc, S0):
    """Intermediates of one chunk of the per-channel chunk algebra (fp64)."""
    n = Kc.shape[0]
    G = np.cumsum(gc, axis=0)                                          # (n, K)
    i, j = np.indices((n, n))
    expo = np.where((i >= j)[:, :, None], G[:, None, :] - G[None, :, :], -np.inf)
    E = np.exp(expo)                                                   # exp(G_ic - G_jc), 0 above
    KE = Kc[None, :, :] * E                                            # k_jc E_ijc
    Ap = np.where(i > j, np.einsum("ic,ijc->ij", Kc, KE), 0.0)          # A without beta
    A = bc[:, None] * Ap
    P = np.einsum("ic,ijc->ij", Q, KE)
    Tm = solve_triangular(np.eye(n) + A, np.eye(n), lower=True, unit_diagonal=True)
    Gam = np.exp(G)
    KG, QG = Gam * Kc, Gam * Q
    U = Vc - KG @ S0                                                   # V - (exp(G) o K) S0
    R = bc[:, None] * U
    Delta = Tm @ R
    Dn = np.exp(G[-1][None, :] - G)                                    # exp(G_n - G)
    Kt = Dn * Kc
    gn = np.exp(G[-1])
    S1 = gn[:, None] * S0 + Kt.T @ Delta
    return dict(G=G, E=E, Ap=Ap, A=A, P=P, Tm=Tm, Gam=Gam, KG=KG, QG=QG, U=U, R=R, Delta=Delta,
                Dn=Dn, Kt=Kt, gn=gn, S0=S0, S1=S1, lower=(i >= j), strict=(i > j))


def kda_chunk_fwd_head(q, k, v, g, beta, scale, S0=None, chunk=64):
    """kda_fwd_head evaluated chunk by chunk.  Per chunk of n <= chunk tokens
    with start state S0 and the per-channel running sums G_i = g_1 + ... + g_i
    (vectors of K):
        A_ij  = beta_i sum_c k_ic k_jc exp(G_ic - G_jc)   for j < i, else 0
        P_ij  =        sum_c q_ic k_jc exp(G_ic - G_jc)   for j <= i, else 0
        Tm    = (I + A)^-1
        Delta = Tm [beta o (V - (exp(G) o K) S0)]
        O     = scale [(exp(G) o Q) S0 + P Delta]
        S1    = diag(exp(G_n)) S0 + (exp(G_n - G) o K)^T Delta
    (exp(G) o K scales k_ic by exp(G_ic)).  Every pair's exponent is masked to
    j <= i before exp, so it is <= 0 for g <= 0.  Returns (o, S) in fp64."""
    q, k, v, g, beta = (np.asarray(x, np.float64) for x in (q, k, v, g, beta))
    T, K = k.shape
    V = v.shape[1]
    S = np.zeros((K, V)) if S0 is None else np.array(S0, dtype=np.float64)
    o = np.zeros((T, V))
    for c0 in range(0, T, chunk):
        sl = slice(c0, min(T, c0 + chunk))
        f = _kda_chunk(q[sl], k[sl], v[sl], g[sl], beta[sl], S)
        o[sl] = scale * (f["QG"] @ S + f["P"] @ f["Delta"])
        S = f["S1"]
    return o, S


def kda_chunk_bwd_head(q, k, v, g, beta, scale, S0, dO, dS_final, chunk=64):
    """Reverse mode of kda_chunk_fwd_head: chunks from last to first, carrying
    dS (the gradient with respect to the chunk-end state).  Per chunk, in
    reverse order of the forward steps:
      O = scale [QG S0 + P Delta]      dQG = scale dO S0^T, dS0 = scale QG^T dO,
                                       dP = scale dO Delta^T (j <= i), dDelta = scale P^T dO
      S1 = diag(gn) S0 + Kt^T Delta    dS0 += diag(gn) dS, dG_n += gn o rowsum(dS o S0),
                                       dKt = Delta dS^T, dDelta += Kt dS
      Kt = exp(G_n - G) o K            dK += dKt o exp(G_n - G); X = dKt o Kt: dG_n += colsum X, dG -= X
      Delta = Tm R                     dR = Tm^T dDelta, dA = -dR Delta^T (j < i)
      R = beta o (V - KG S0)           dV = beta o dR, dbeta += rowsum(dR o U),
                                       dKG = -(beta o dR) S0^T, dS0 -= KG^T (beta o dR)
      KG = exp(G) o K, QG = exp(G) o Q dK += dKG o exp(G), dQ += dQG o exp(G), dG += dKG o KG + dQG o QG
      A = beta o A', A'_ij = sum_c k_ic k_jc E_ijc (j < i)
                                       dbeta += rowsum(dA o A'); W = beta o dA:
                                       dk_i += sum_j W_ij k_j o E_ij, dk_j += sum_i W_ij k_i o E_ij
      P_ij = sum_c q_ic k_jc E_ijc     dq_i += sum_j dP_ij k_j o E_ij, dk_j += sum_i dP_ij q_i o E_ij
      E_ijc = exp(G_ic - G_jc)         Y_ijc = (W_ij k_ic + dP_ij q_ic) k_jc E_ijc:
                                       dG_i += sum_j Y_ij, dG_j -= sum_i Y_ij
      G = cumsum(g)                    dg = reverse running sum of dG, per channel
    Returns dict of dq, dk (T, K), dv (T, V), dg (T, K), dbeta (T,), dS0 (K, V)."""
    q, k, v, g, beta, dO = (np.asarray(x, np.float64) for x in (q, k, v, g, beta, dO))
    T, K = k.shape
    V = v.shape[1]
    S = np.zeros((K, V)) if S0 is None else np.array(S0, dtype=np.float64)
    chunks = []
    for c0 in range(0, T, chunk):
        sl = slice(c0, min(T, c0 + chunk))
        f = _kda_chunk(q[sl], k[sl], v[sl], g[sl], beta[sl], S)
        chunks.append((sl, f))
        S = f["S1"]
    out = dict(dq=np.zeros((T, K)), dk=np.zeros((T, K)), dv=np.zeros((T, V)), dg=np.zeros((T, K)),
               dbeta=np.zeros(T), dS0=None)
    dS = np.zeros((K, V)) if dS_final is None else np.array(dS_final, dtype=np.float64)
    for sl, f in reversed(chunks):
        Q, Kc, bc, dOc, S0c = q[sl], k[sl], beta[sl], dO[sl], f["S0"]
        E = f["E"]
        # output
        dQG = scale * dOc @ S0c.T
        dS0 = scale * f["QG"].T @ dOc
        dP = np.where(f["lower"], scale * dOc @ f["Delta"].T, 0.0)
        dDelta = scale * f["P"].T @ dOc
        # state update
        dS0 += f["gn"][:, None] * dS
        dG = np.zeros_like(f["G"])
        dG[-1] += f["gn"] * np.sum(dS * S0c, axis=1)
        dKt = f["Delta"] @ dS.T
        dDelta += f["Kt"] @ dS
        dK = dKt * f["Dn"]
        X = dKt * f["Kt"]
        dG[-1] += X.sum(axis=0)
        dG -= X
        # triangular solve and residual
        dR = f["Tm"].T @ dDelta
        dA = np.where(f["strict"], -dR @ f["Delta"].T, 0.0)
        dv = bc[:, None] * dR
        dbeta = np.sum(dR * f["U"], axis=1)
        dKG = -(bc[:, None] * dR) @ S0c.T
        dS0 -= f["KG"].T @ (bc[:, None] * dR)
        dK += dKG * f["Gam"]
        dQ = dQG * f["Gam"]
        dG += dKG * f["KG"] + dQG * f["QG"]
        # the two decayed sums
        dbeta += np.sum(dA * f["Ap"], axis=1)
        W = bc[:, None] * dA
        dK += np.einsum("ij,jc,ijc->ic", W, Kc, E) + np.einsum("ij,ic,ijc->jc", W, Kc, E)
        dQ += np.einsum("ij,jc,ijc->ic", dP, Kc, E)
        dK += np.einsum("ij,ic,ijc->jc", dP, Q, E)
        Y = (W[:, :, None] * Kc[:, None, :] + dP[:, :, None] * Q[:, None, :]) * Kc[None, :, :] * E
        dG += Y.sum(axis=1) - Y.sum(axis=0)
        out["dq"][sl] = dQ
        out["dk"][sl] = dK
        out["dv"][sl] = dv
        out["dbeta"][sl] = dbeta
        out["dg"][sl] = np.cumsum(dG[::-1], axis=0)[::-1]
        dS = dS0
    out["dS0"] = dS
    return out


def kda_bwd_head(q, k, v, g, beta, scale, S0, dO, dS_final, checkpoint=64):
    """Reverse mode of kda_fwd_head, token by token from t = T down to 1, with
    the state recomputed forward from checkpoints every `checkpoint` tokens.
    Per token (S' = diag(exp(g_t)) S_{t-1}, e = v_t - S'^T k_t,
    S_t = S' + beta_t k_t e^T, o_t = scale S_t^T q_t), with dS the gradient
    with respect to S_t:
        dS    += scale q_t dO_t^T;        dq_t = scale S_t dO_t
        dbeta_t = k_t^T dS e;             de = beta_t dS^T k_t
        dv_t  = de;                        dk_t = beta_t dS e - S' de
        dS'   = dS - k_t de^T;             dg_t = rowsum(dS' o S')   (per key channel)
        dS_{t-1} = diag(exp(g_t)) dS'
    Returns dict of dq, dk (T, K), dv (T, V), dg (T, K), dbeta (T,), dS0 (K, V)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(g, np.float64)
    beta = np.asarray(beta, np.float64)
    dO = np.asarray(dO, np.float64)
    T, K = k.shape
    V = v.shape[1]
    S = np.zeros((K, V)) if S0 is None else np.array(S0, dtype=np.float64)
    # forward: the state at the start of every checkpoint segment
    starts = []
    for t in range(T):
        if t % checkpoint == 0:
            starts.append(S.copy())
        S = np.exp(g[t])[:, None] * S
        S = S + beta[t] * np.outer(k[t], v[t] - S.T @ k[t])
    out = dict(dq=np.zeros((T, K)), dk=np.zeros((T, K)), dv=np.zeros((T, V)), dg=np.zeros((T, K)),
               dbeta=np.zeros(T), dS0=None)
    dS = np.zeros((K, V)) if dS_final is None else np.array(dS_final, dtype=np.float64)
    for si in range(len(starts) - 1, -1, -1):
        t0 = si * checkpoint
        t1 = min(T, t0 + checkpoint)
        # recompute S'_t and S_t inside the segment
        Sp, St = [], []
        S = starts[si].copy()
        for t in range(t0, t1):
            S = np.exp(g[t])[:, None] * S
            Sp.append(S.copy())
            S = S + beta[t] * np.outer(k[t], v[t] - S.T @ k[t])
            St.append(S.copy())
        for t in range(t1 - 1, t0 - 1, -1):
            P, Sn = Sp[t - t0], St[t - t0]
            dS = dS + scale * np.outer(q[t], dO[t])
            out["dq"][t] = scale * (Sn @ dO[t])
            e = v[t] - P.T @ k[t]
            out["dbeta"][t] = k[t] @ dS @ e
            de = beta[t] * (dS.T @ k[t])
            out["dv"][t] = de
            out["dk"][t] = beta[t] * (dS @ e) - P @ de
            dSp = dS - np.outer(k[t], de)
            out["dg"][t] = np.sum(dSp * P, axis=1)
            dS = np.exp(g[t])[:, None] * dSp
    out["dS0"] = dS
    return out
