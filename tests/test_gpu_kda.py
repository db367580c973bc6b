"""The per-channel-gate (KDA) token-serial forward against the fp64 KDA
oracle, and against the scalar-gate path when every channel shares one gate."""

import numpy as np
import pytest

from linear_attention_sequence_chunked_gb300 import gdn
from linear_attention_sequence_chunked_gb300 import workloads as W
from oracle import kda
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu


def _case(B, T, H, dk, dv, seed, seqlens=None):
    rng = np.random.default_rng(seed)
    n_tok = sum(seqlens) if seqlens is not None else T
    Bd = 1 if seqlens is not None else B
    q = W.f32_to_bf16_bits(rng.standard_normal((Bd, n_tok, H, dk)).astype(np.float32))
    kr = rng.standard_normal((Bd, n_tok, H, dk)).astype(np.float32)
    kr /= np.linalg.norm(kr, axis=-1, keepdims=True)
    k = W.f32_to_bf16_bits(kr)
    v = W.f32_to_bf16_bits(rng.standard_normal((Bd, n_tok, H, dv)).astype(np.float32))
    # per-channel log decays in (-5, 0): the bounded form lower * sigmoid(x)
    g = (-5.0 / (1.0 + np.exp(-rng.standard_normal((Bd, n_tok, H, dk)) - 2.0))).astype(np.float32)
    beta = W.f32_to_bf16_bits((1.0 / (1.0 + np.exp(-rng.standard_normal((Bd, n_tok, H))))).astype(np.float32))
    n_seq = len(seqlens) if seqlens is not None else B
    s0 = (rng.standard_normal((n_seq, H, dk, dv)) / np.sqrt(dk)).astype(np.float32)
    cu = None
    if seqlens is not None:
        cu = np.zeros(len(seqlens) + 1, np.int32)
        cu[1:] = np.cumsum(seqlens)
    return q, k, v, g, beta, s0, cu


def _run(torch, fn, q, k, v, g, beta, s0, cu, scale):
    Bd, n_tok, H, dk = q.shape
    dv = v.shape[3]
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa: E731
    bf = lambda x: d(x.view(np.int16)).view(torch.bfloat16)  # noqa: E731
    n_seq = s0.shape[0]
    out = torch.empty((Bd, n_tok, H, dv), dtype=torch.bfloat16, device="cuda")
    fs = torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device="cuda")
    B = n_seq if cu is not None else Bd
    fn(bf(q), bf(k), bf(v), d(g), bf(beta), scale, d(s0), None if cu is None else d(cu), out, fs,
       B, n_tok, H, dk, dv)
    st = gdn.gdn_get_last_device_error()
    assert st == 0, gdn.gdn_status_string(st)
    torch.cuda.synchronize()
    return G.bf16_to_np(out), fs.cpu().numpy()


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (128, 256)])
def test_kda_matches_oracle(dk, dv):
    import torch
    q, k, v, g, beta, s0, cu = _case(2, 150, 2, dk, dv, seed=dk + dv)
    scale = dk ** -0.5
    o, S = _run(torch, gdn.gdn_kda_recurrent_fwd, q, k, v, g, beta, s0, cu, scale)
    f = W.bf16_bits_to_f32
    o_ref, S_ref = kda.kda_fwd(f(q), f(k), f(v), g, f(beta), scale, s0)
    G.compare(o, o_ref, G.TOL_RMS_IID, G.TOL_MAX_IID, "kda out")
    G.compare(S, S_ref, 1e-5, None, "kda state")


def test_kda_varlen_matches_oracle():
    import torch
    lens = [1, 70, 0, 129]
    q, k, v, g, beta, s0, cu = _case(1, 0, 3, 128, 64, seed=4, seqlens=lens)
    o, S = _run(torch, gdn.gdn_kda_recurrent_fwd, q, k, v, g, beta, s0, cu, 0.1)
    f = W.bf16_bits_to_f32
    o_ref, S_ref = kda.kda_fwd(f(q), f(k), f(v), g, f(beta), 0.1, s0, cu)
    G.compare(o, o_ref, G.TOL_RMS_IID, G.TOL_MAX_IID, "kda varlen out")
    for s in range(len(lens)):
        G.compare(S[s], S_ref[s], 1e-5, None, f"kda varlen state {s}")
    assert np.array_equal(S[2], s0[2])


def test_kda_with_equal_channels_is_the_scalar_path_bitwise():
    import torch
    q, k, v, g, beta, s0, cu = _case(2, 90, 2, 128, 64, seed=9)
    g1 = np.ascontiguousarray(g[..., 0])
    gk = np.ascontiguousarray(np.repeat(g1[..., None], 128, axis=-1))
    o1, S1 = _run(torch, gdn.gdn_kda_recurrent_fwd, q, k, v, gk, beta, s0, cu, 0.2)
    o2, S2 = _run(torch, gdn.gdn_recurrent_fwd, q, k, v, g1, beta, s0, cu, 0.2)
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)


# ---------------------------------------------------------------------------
# the chunked forward (gdn_kda_chunk_fwd)
# ---------------------------------------------------------------------------

TOL_STATE_FP32 = 1e-4   # fp32 chunk arithmetic throughout; the state is never rounded to bf16


def _check_against_oracle(o, S, q, k, v, g, beta, s0, cu, scale, what):
    f = W.bf16_bits_to_f32
    o_ref, S_ref = kda.kda_fwd(f(q), f(k), f(v), g, f(beta), scale, s0, cu)
    G.compare(o, o_ref, G.TOL_RMS_IID, G.TOL_MAX_IID, what + " out")
    for s in range(S.shape[0]):
        G.compare(S[s], S_ref[s], TOL_STATE_FP32, None, f"{what} state {s}")


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 128), (128, 256)])
def test_kda_chunk_matches_oracle(dk, dv):
    """Three chunks per sequence, the last one ragged (150 = 2 x 64 + 22)."""
    import torch
    q, k, v, g, beta, s0, cu = _case(2, 150, 2, dk, dv, seed=100 + dk + dv)
    scale = dk ** -0.5
    o, S = _run(torch, gdn.gdn_kda_chunk_fwd, q, k, v, g, beta, s0, cu, scale)
    _check_against_oracle(o, S, q, k, v, g, beta, s0, cu, scale, "kda chunk")


def test_kda_chunk_varlen_matches_oracle():
    """Packed sequences of 1, 63, 64, 65, 0 and 200 tokens: resets at every
    boundary, chunks never straddle sequences, an empty sequence passes its
    initial state through unchanged."""
    import torch
    lens = [1, 63, 64, 65, 0, 200]
    q, k, v, g, beta, s0, cu = _case(1, 0, 2, 128, 64, seed=12, seqlens=lens)
    o, S = _run(torch, gdn.gdn_kda_chunk_fwd, q, k, v, g, beta, s0, cu, 0.1)
    _check_against_oracle(o, S, q, k, v, g, beta, s0, cu, 0.1, "kda chunk varlen")
    assert np.array_equal(S[4], s0[4])


def test_kda_chunk_strong_per_channel_decay():
    """Per-channel log decays down to -40 per token: inside a chunk the
    exponents G_ic - G_jc reach about -2500, far below the fp32 range of exp;
    formed as masked differences they underflow to 0 and never overflow."""
    import torch
    q, k, v, g, beta, s0, cu = _case(1, 200, 2, 128, 128, seed=13)
    g = (g * 8.0).astype(np.float32)
    scale = 128 ** -0.5
    o, S = _run(torch, gdn.gdn_kda_chunk_fwd, q, k, v, g, beta, s0, cu, scale)
    assert np.isfinite(o).all() and np.isfinite(S).all()
    _check_against_oracle(o, S, q, k, v, g, beta, s0, cu, scale, "kda chunk strong decay")


def test_kda_chunk_agrees_with_token_serial_and_repeats_bitwise():
    """The chunked and the token-serial kernels agree within the output
    tolerance; a second launch of the chunked kernel is bitwise the first."""
    import torch
    q, k, v, g, beta, s0, cu = _case(2, 300, 3, 128, 128, seed=14)
    o1, S1 = _run(torch, gdn.gdn_kda_chunk_fwd, q, k, v, g, beta, s0, cu, 0.09)
    o2, S2 = _run(torch, gdn.gdn_kda_chunk_fwd, q, k, v, g, beta, s0, cu, 0.09)
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)
    o3, S3 = _run(torch, gdn.gdn_kda_recurrent_fwd, q, k, v, g, beta, s0, cu, 0.09)
    G.compare(o1, o3, G.TOL_RMS_IID, G.TOL_MAX_IID, "chunked vs token-serial out")
    G.compare(S1, S3, TOL_STATE_FP32, None, "chunked vs token-serial state")


def test_kda_chunk_zero_length():
    import torch
    q, k, v, g, beta, s0, cu = _case(2, 0, 2, 64, 64, seed=15)
    o, S = _run(torch, gdn.gdn_kda_chunk_fwd, q, k, v, g, beta, s0, cu, 0.125)
    assert o.size == 0 and np.array_equal(S, s0)


def test_kda_chunk_long_sequence_sampled_heads():
    """T = 4096 (64 chunks in series), d_k = d_v = 128, through the wrapper
    that allocates the outputs; every head against the oracle."""
    import torch
    q, k, v, g, beta, s0, cu = _case(1, 4096, 2, 128, 128, seed=16)
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa: E731
    bf = lambda x: d(x.view(np.int16)).view(torch.bfloat16)  # noqa: E731
    out, fs = gdn.chunk_kda_fwd(bf(q), bf(k), bf(v), d(g), bf(beta), scale=128 ** -0.5, initial_state=d(s0))
    st = gdn.gdn_get_last_device_error()
    assert st == 0, gdn.gdn_status_string(st)
    torch.cuda.synchronize()
    _check_against_oracle(G.bf16_to_np(out), fs.cpu().numpy(), q, k, v, g, beta, s0, cu, 128 ** -0.5,
                          "kda chunk T=4096")
