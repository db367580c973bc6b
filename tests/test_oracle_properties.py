"""Property tests of the fp64 oracle over random shapes (hypothesis; CPU
only): three independent formulations of the same operator agree on any
input -- the per-token recurrence (C), the chunked WY algebra at any chunk
length, and the segment composition at any cut points -- the
per-channel-gate recurrence reduces to the scalar one when its channels
are equal, and its chunk algebra equals its token loop."""

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

from oracle import chunked, kda, recurrence, segments  # noqa: E402

SETTINGS = settings(max_examples=25, deadline=None, derandomize=True)


def _lib():
    return recurrence._load()


def _head(draw_seed, T, K, V, beta_max, g_low):
    r = np.random.default_rng(draw_seed)
    q = r.standard_normal((T, K))
    k = r.standard_normal((T, K))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = r.standard_normal((T, V))
    g = r.uniform(g_low, 0.0, T)
    beta = r.uniform(0.0, beta_max, T)
    S0 = r.standard_normal((K, V))
    return q, k, v, g, beta, S0


def _rel(x, r):
    return float(np.max(np.abs(np.asarray(x) - np.asarray(r))) / max(np.max(np.abs(r)), 1e-300))


shapes = st.tuples(st.integers(1, 150), st.integers(1, 9), st.integers(1, 7))


@SETTINGS
@given(shape=shapes, chunk=st.integers(1, 70), seed=st.integers(0, 2**31 - 1),
       beta_max=st.sampled_from([1.0, 2.0]), g_low=st.sampled_from([-0.05, -0.5, -4.0]))
def test_chunked_algebra_equals_recurrence(shape, chunk, seed, beta_max, g_low):
    T, K, V = shape
    q, k, v, g, beta, S0 = _head(seed, T, K, V, beta_max, g_low)
    o1, S1 = _lib().fwd_head(q, k, v, g, beta, 0.7, S0)
    o2, S2, _ = chunked.fwd_head(q, k, v, g, beta, 0.7, S0, chunk=chunk)
    assert _rel(o2, o1) < 1e-10 and _rel(S2, S1) < 1e-10


@SETTINGS
@given(shape=shapes, seed=st.integers(0, 2**31 - 1), data=st.data())
def test_segment_composition_equals_recurrence(shape, seed, data):
    T, K, V = shape
    q, k, v, g, beta, S0 = _head(seed, T, K, V, 2.0, -0.5)
    cuts = sorted(set(data.draw(st.lists(st.integers(1, max(1, T - 1)), max_size=8)))) if T > 1 else []
    lib = _lib()
    o1, S1 = lib.fwd_head(q, k, v, g, beta, 0.4, S0)
    o2, S2, _ = segments.segmented_fwd(lib.fwd_head, q, k, v, g, beta, 0.4, S0, cuts)
    assert _rel(o2, o1) < 1e-11 and _rel(S2, S1) < 1e-11


@SETTINGS
@given(shape=shapes, seed=st.integers(0, 2**31 - 1))
def test_per_channel_gate_with_equal_channels_is_the_scalar_gate(shape, seed):
    T, K, V = shape
    q, k, v, g, beta, S0 = _head(seed, T, K, V, 2.0, -0.5)
    o1, S1 = _lib().fwd_head(q, k, v, g, beta, 0.3, S0)
    o2, S2 = kda.kda_fwd_head(q, k, v, np.repeat(g[:, None], K, axis=1), beta, 0.3, S0)
    assert _rel(o2, o1) < 1e-12 and _rel(S2, S1) < 1e-12


@SETTINGS
@given(shape=shapes, chunk=st.integers(1, 70), seed=st.integers(0, 2**31 - 1),
       beta_max=st.sampled_from([1.0, 2.0]), g_low=st.sampled_from([-0.05, -0.5, -4.0, -40.0]))
def test_per_channel_chunk_algebra_equals_its_token_loop(shape, chunk, seed, beta_max, g_low):
    """Per-channel decays drawn independently per token and key channel, down
    to -40 per token (exponents far below the fp64 range of exp inside a
    chunk)."""
    T, K, V = shape
    r = np.random.default_rng(seed)
    q, k, v, _, beta, S0 = _head(seed, T, K, V, beta_max, g_low)
    g = r.uniform(g_low, 0.0, (T, K))
    o1, S1 = kda.kda_fwd_head(q, k, v, g, beta, 0.6, S0)
    o2, S2 = kda.kda_chunk_fwd_head(q, k, v, g, beta, 0.6, S0, chunk=chunk)
    assert np.isfinite(o2).all() and np.isfinite(S2).all()
    assert _rel(o2, o1) < 1e-10 and _rel(S2, S1) < 1e-10


@SETTINGS
@given(shape=st.tuples(st.integers(1, 80), st.integers(1, 6), st.integers(1, 5)), chunk=st.integers(1, 70),
       seed=st.integers(0, 2**31 - 1), g_low=st.sampled_from([-0.05, -0.5, -4.0, -40.0]))
def test_per_channel_chunked_reverse_mode_equals_token_reverse_mode(shape, chunk, seed, g_low):
    T, K, V = shape
    r = np.random.default_rng(seed)
    q, k, v, _, beta, S0 = _head(seed, T, K, V, 2.0, g_low)
    g = r.uniform(g_low, 0.0, (T, K))
    dO = r.standard_normal((T, V))
    dSf = r.standard_normal((K, V))
    a = kda.kda_bwd_head(q, k, v, g, beta, 0.6, S0, dO, dSf)
    b = kda.kda_chunk_bwd_head(q, k, v, g, beta, 0.6, S0, dO, dSf, chunk=chunk)
    for name in a:
        assert np.isfinite(b[name]).all(), name
        assert _rel(b[name], a[name]) < 1e-9, name


@SETTINGS
@given(shape=shapes, seed=st.integers(0, 2**31 - 1), data=st.data())
def test_per_channel_segment_composition_equals_token_loop(shape, seed, data):
    T, K, V = shape
    r = np.random.default_rng(seed)
    q, k, v, _, beta, S0 = _head(seed, T, K, V, 2.0, -0.5)
    g = r.uniform(-0.5, 0.0, (T, K))
    cuts = sorted(set(data.draw(st.lists(st.integers(1, max(1, T - 1)), max_size=8)))) if T > 1 else []
    o1, S1 = kda.kda_fwd_head(q, k, v, g, beta, 0.4, S0)
    o2, S2, _ = segments.segmented_fwd(kda.kda_fwd_head, q, k, v, g, beta, 0.4, S0, cuts)
    assert _rel(o2, o1) < 1e-10 and _rel(S2, S1) < 1e-10
