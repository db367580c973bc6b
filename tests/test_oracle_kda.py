"""Pins of the fp64 per-channel-gate (KDA) oracle: equal channels reduce to
the scalar-gate C oracle, beta = 0 is pure per-channel decay, the T = 1
closed form, the chunked formulation equals the token loop, the reverse mode
matches central finite differences and (equal channels) the scalar C
oracle's reverse mode, and planted mistakes that the pins catch."""

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



def _rel(x, r):
    return float(np.max(np.abs(x - r)) / max(np.max(np.abs(r)), 1e-300))


@pytest.mark.parametrize("T,chunk", [(1, 64), (37, 64), (64, 64), (65, 64), (150, 64), (150, 16), (41, 5)])
def test_chunked_equals_token_loop(T, chunk):
    """The per-channel chunk algebra reaches the token loop's result: one
    token, a ragged single chunk, exact multiples, a ragged tail, and chunk
    sizes that cut the sequence into many pieces."""
    q, k, v, g, beta, S0 = _head(T, 6, 5, 10 + T + chunk)
    beta = beta * 2.0
    o_ref, S_ref = kda.kda_fwd_head(q, k, v, g, beta, 0.45, S0)
    o, S = kda.kda_chunk_fwd_head(q, k, v, g, beta, 0.45, S0, chunk=chunk)
    assert _rel(o, o_ref) < 1e-12 and _rel(S, S_ref) < 1e-12, (_rel(o, o_ref), _rel(S, S_ref))


def test_chunked_equals_token_loop_wider_heads():
    q, k, v, g, beta, S0 = _head(130, 16, 12, 21)
    o_ref, S_ref = kda.kda_fwd_head(q, k, v, g, beta, 0.25, S0)
    o, S = kda.kda_chunk_fwd_head(q, k, v, g, beta, 0.25, S0)
    assert _rel(o, o_ref) < 1e-12 and _rel(S, S_ref) < 1e-12


def _factorised_chunk_head(q, k, v, g, beta, scale, S0, chunk=64):
    """A planted mistake: the decay of a pair written as exp(G_i) exp(-G_j),
    without masking before exp."""
    T, K = k.shape
    S = np.array(S0, dtype=np.float64)
    o = np.zeros((T, v.shape[1]))
    with np.errstate(over="ignore", invalid="ignore"):
        for c0 in range(0, T, chunk):
            sl = slice(c0, min(T, c0 + chunk))
            Q, Kc, Vc, b = q[sl], k[sl], v[sl], beta[sl]
            n = Kc.shape[0]
            G = np.cumsum(g[sl], axis=0)
            up, down = np.exp(G) * Kc, np.exp(-G) * Kc
            i, j = np.indices((n, n))
            A = np.where(i > j, b[:, None] * (up @ down.T), 0.0)
            P = np.where(i >= j, (np.exp(G) * Q) @ down.T, 0.0)
            Tm = np.linalg.inv(np.eye(n) + A)
            Delta = Tm @ (b[:, None] * (Vc - up @ S))
            o[sl] = scale * ((np.exp(G) * Q) @ S + P @ Delta)
            S = np.exp(G[-1])[:, None] * S + (np.exp(G[-1][None, :] - G) * Kc).T @ Delta
    return o, S


def test_strong_decay_needs_the_masked_exponent():
    """Per-channel log decays down to -40 per token: inside a 64-token chunk
    G reaches about -2500.  The masked form stays finite and exact; writing a
    pair's decay as exp(G_i) exp(-G_j) overflows."""
    q, k, v, g, beta, S0 = _head(128, 6, 5, 22)
    g = g * 80.0
    o_ref, S_ref = kda.kda_fwd_head(q, k, v, g, beta, 0.5, S0)
    o, S = kda.kda_chunk_fwd_head(q, k, v, g, beta, 0.5, S0)
    assert np.isfinite(o).all() and np.isfinite(S).all()
    assert _rel(o, o_ref) < 1e-12 and _rel(S, S_ref) < 1e-12
    o_bad, S_bad = _factorised_chunk_head(q, k, v, g, beta, 0.5, S0)
    assert not (np.isfinite(o_bad).all() and _rel(o_bad, o_ref) < 1e-6)


def test_chunked_planted_mistakes_are_caught():
    """The chunked pin catches a scalar gate (the per-channel decays replaced
    by their mean), a causal score without its diagonal, and the gram with its
    diagonal kept."""
    q, k, v, g, beta, S0 = _head(100, 6, 5, 23)
    o_ref, S_ref = kda.kda_fwd_head(q, k, v, g, beta, 0.5, S0)
    gm = np.repeat(g.mean(axis=1, keepdims=True), 6, axis=1)
    o, S = kda.kda_chunk_fwd_head(q, k, v, gm, beta, 0.5, S0)
    assert _rel(o, o_ref) > 1e-6

    def variant(drop_p_diag, keep_a_diag):
        T = 100
        S = np.array(S0)
        o = np.zeros((T, 5))
        for c0 in range(0, T, 64):
            sl = slice(c0, min(T, c0 + 64))
            Q, Kc, Vc, b = q[sl], k[sl], v[sl], beta[sl]
            n = Kc.shape[0]
            G = np.cumsum(g[sl], axis=0)
            i, j = np.indices((n, n))
            expo = np.where((i >= j)[:, :, None], G[:, None, :] - G[None, :, :], -np.inf)
            KE = Kc[None, :, :] * np.exp(expo)
            A = np.where((i >= j) if keep_a_diag else (i > j), b[:, None] * np.einsum("ic,ijc->ij", Kc, KE), 0.0)
            P = np.einsum("ic,ijc->ij", Q, KE)
            if drop_p_diag:
                P = np.where(i > j, P, 0.0)
            Tm = np.linalg.inv(np.eye(n) + A)
            Delta = Tm @ (b[:, None] * (Vc - (np.exp(G) * Kc) @ S))
            o[sl] = 0.5 * ((np.exp(G) * Q) @ S + P @ Delta)
            S = np.exp(G[-1])[:, None] * S + (np.exp(G[-1][None, :] - G) * Kc).T @ Delta
        return o, S

    for flags in ((False, False), (True, False), (False, True)):
        o, S = variant(*flags)
        if flags == (False, False):
            assert _rel(o, o_ref) < 1e-12   # the variant itself is the right algebra
        else:
            assert _rel(o, o_ref) > 1e-6, flags



def _fd_check(bwd, T, K, V, seed, checkpoint=64):
    q, k, v, g, beta, S0 = _head(T, K, V, seed)
    beta = beta * 2.0
    r = np.random.default_rng(seed + 1)
    dO = r.standard_normal((T, V))
    dSf = r.standard_normal((K, V))
    scale = 0.7

    def loss(args):
        o, S = kda.kda_fwd_head(*args[:5], scale, args[5])
        return float(np.sum(o * dO) + np.sum(S * dSf))

    grads = bwd(q, k, v, g, beta, scale, S0, dO, dSf, checkpoint=checkpoint)
    args = [q, k, v, g, beta, S0]
    worst = {}
    for ai, name in enumerate(["dq", "dk", "dv", "dg", "dbeta", "dS0"]):
        fd = np.zeros_like(args[ai])
        for idx in np.ndindex(args[ai].shape):
            ap = [a.copy() for a in args]
            am = [a.copy() for a in args]
            ap[ai][idx] += 1e-6
            am[ai][idx] -= 1e-6
            fd[idx] = (loss(ap) - loss(am)) / 2e-6
        worst[name] = _rel(grads[name], fd)
    return worst


@pytest.mark.parametrize("T,K,V,checkpoint", [(7, 3, 4, 64), (8, 4, 3, 3), (1, 2, 2, 64)])
def test_reverse_mode_matches_finite_differences(T, K, V, checkpoint):
    """Every gradient (dg per key channel) against central differences of
    L = <o, dO> + <S_T, dS_T>, with and without checkpoint segments."""
    worst = _fd_check(kda.kda_bwd_head, T, K, V, 30 + T, checkpoint)
    assert all(e < 1e-7 for e in worst.values()), worst


def test_reverse_mode_with_equal_channels_is_the_scalar_reverse_mode(lib):
    """All channels equal: every gradient equals the scalar-gate C oracle's,
    with dg summed over the key channels."""
    q, k, v, g, beta, S0 = _head(150, 6, 5, 40)
    gs = g[:, 0]
    r = np.random.default_rng(41)
    dO = r.standard_normal((150, 5))
    dSf = r.standard_normal((6, 5))
    a = kda.kda_bwd_head(q, k, v, np.repeat(gs[:, None], 6, axis=1), beta * 2.0, 0.4, S0, dO, dSf)
    b = lib.bwd_head(q, k, v, gs, beta * 2.0, 0.4, S0, dO, dSf)
    for name in ("dq", "dk", "dv", "dbeta", "dS0"):
        assert _rel(a[name], b[name]) < 1e-12, name
    assert _rel(a["dg"].sum(axis=1), b["dg"]) < 1e-12


def test_reverse_mode_planted_mistake_is_caught():
    """A per-channel gate gradient summed over the value columns of the state
    before the decay (dS' o S_{t-1} instead of dS' o S') breaks the
    finite-difference pin."""
    def wrong(q, k, v, g, beta, scale, S0, dO, dSf, checkpoint=64):
        out = kda.kda_bwd_head(q, k, v, g, beta, scale, S0, dO, dSf, checkpoint)
        out["dg"] = out["dg"] * np.exp(-g)    # the pre-decay state's rows
        return out
    worst = _fd_check(wrong, 7, 3, 4, 37)
    assert worst["dg"] > 1e-6 and worst["dq"] < 1e-7


CHUNK_BWD_CASES = [(7, 3, 4, 64, -0.5), (150, 6, 5, 64, -0.5), (97, 4, 8, 16, -0.5), (41, 5, 3, 5, -4.0),
                   (128, 6, 5, 64, -40.0), (1, 2, 2, 64, -0.5)]


def _bwd_inputs(T, K, V, g_low, seed):
    r = np.random.default_rng(seed)
    q = r.standard_normal((T, K))
    k = r.standard_normal((T, K))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = r.standard_normal((T, V))
    g = r.uniform(g_low, 0.0, (T, K))
    beta = r.uniform(0.0, 2.0, T)
    S0 = r.standard_normal((K, V))
    return q, k, v, g, beta, S0, r.standard_normal((T, V)), r.standard_normal((K, V))


@pytest.mark.parametrize("T,K,V,chunk,g_low", CHUNK_BWD_CASES)
def test_chunked_reverse_mode_equals_token_reverse_mode(T, K, V, chunk, g_low):
    """The reverse mode of the per-channel chunk algebra (derived step by step
    through the chunk's intermediates) gives the token loop's gradients:
    ragged chunks, chunk sizes 64 / 16 / 5, decays down to -40 per token."""
    q, k, v, g, beta, S0, dO, dSf = _bwd_inputs(T, K, V, g_low, 50 + T)
    a = kda.kda_bwd_head(q, k, v, g, beta, 0.6, S0, dO, dSf)
    b = kda.kda_chunk_bwd_head(q, k, v, g, beta, 0.6, S0, dO, dSf, chunk=chunk)
    for name in a:
        assert _rel(b[name], a[name]) < 1e-11, (name, _rel(b[name], a[name]))


MUTATIONS = [
    ("gram column-role key gradient dropped",
     ' + np.einsum("ij,ic,ijc->jc", W, Kc, E)', ""),
    ("decay-exponent gradient of the earlier token dropped",
     "dG += Y.sum(axis=1) - Y.sum(axis=0)", "dG += Y.sum(axis=1)"),
    ("gram gradient kept on the diagonal",
     'dA = np.where(f["strict"], -dR @ f["Delta"].T, 0.0)', 'dA = np.where(f["lower"], -dR @ f["Delta"].T, 0.0)'),
    ("gate gradient summed forward instead of backward",
     'out["dg"][sl] = np.cumsum(dG[::-1], axis=0)[::-1]', 'out["dg"][sl] = np.cumsum(dG, axis=0)'),
    ("state-decay gate gradient dropped",
     'dG[-1] += f["gn"] * np.sum(dS * S0c, axis=1)', "pass"),
]


@pytest.mark.parametrize("what,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_chunked_reverse_mode_planted_mistakes_are_caught(what, old, new):
    """Each mistake, planted in a copy of the chunked reverse mode's source,
    breaks its agreement with the token loop's reverse mode."""
    import inspect
    import textwrap
    src = textwrap.dedent(inspect.getsource(kda.kda_chunk_bwd_head))
    assert src.count(old) == 1, what
    ns = dict(vars(kda))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    q, k, v, g, beta, S0, dO, dSf = _bwd_inputs(150, 6, 5, -0.5, 60)
    ref = kda.kda_bwd_head(q, k, v, g, beta, 0.6, S0, dO, dSf)
    bad = ns["kda_chunk_bwd_head"](q, k, v, g, beta, 0.6, S0, dO, dSf, chunk=64)
    assert max(_rel(bad[n], ref[n]) for n in ref) > 1e-6, what
