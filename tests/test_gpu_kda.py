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
