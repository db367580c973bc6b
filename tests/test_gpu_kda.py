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


def _run(torch, fn, q, k, v, g, beta, s0, cu, scale, tp=False):
    """One forward call; with tp, gdn_kda_chunk_fwd gets its workspace (every
    chunk's T and P formed first by the chunk-parallel kernel)."""
    Bd, n_tok, H, dk = q.shape
    dv = v.shape[3]
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa: E731
    bf = lambda x: d(x.view(np.int16)).view(torch.bfloat16)  # noqa: E731
    n_seq = s0.shape[0]
    out = torch.empty((Bd, n_tok, H, dv), dtype=torch.bfloat16, device="cuda")
    fs = torch.empty((n_seq, H, dk, dv), dtype=torch.float32, device="cuda")
    B = n_seq if cu is not None else Bd
    extra = {}
    if tp:
        nbytes = gdn.gdn_kda_chunk_fwd_workspace_size(B, n_tok, H, dk, dv, cu is not None)
        extra = dict(workspace=torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda"),
                     workspace_bytes=nbytes)
    fn(bf(q), bf(k), bf(v), d(g), bf(beta), scale, d(s0), None if cu is None else d(cu), out, fs,
       B, n_tok, H, dk, dv, **extra)
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


@pytest.mark.parametrize("tp", [False, True], ids=["walk", "tp"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128), (128, 256)])
def test_kda_chunk_matches_oracle(dk, dv, tp):
    """Three chunks per sequence, the last one ragged (150 = 2 x 64 + 22); the
    walk that forms T and P itself, and the route that reads them from the
    chunk-parallel kernel's workspace."""
    import torch
    q, k, v, g, beta, s0, cu = _case(2, 150, 2, dk, dv, seed=100 + dk + dv)
    scale = dk ** -0.5
    o, S = _run(torch, gdn.gdn_kda_chunk_fwd, q, k, v, g, beta, s0, cu, scale, tp=tp)
    _check_against_oracle(o, S, q, k, v, g, beta, s0, cu, scale, "kda chunk")


@pytest.mark.parametrize("tp", [False, True], ids=["walk", "tp"])
def test_kda_chunk_varlen_matches_oracle(tp):
    """Packed sequences of 1, 63, 64, 65, 0 and 200 tokens: resets at every
    boundary, chunks never straddle sequences, an empty sequence passes its
    initial state through unchanged."""
    import torch
    lens = [1, 63, 64, 65, 0, 200]
    q, k, v, g, beta, s0, cu = _case(1, 0, 2, 128, 64, seed=12, seqlens=lens)
    o, S = _run(torch, gdn.gdn_kda_chunk_fwd, q, k, v, g, beta, s0, cu, 0.1, tp=tp)
    _check_against_oracle(o, S, q, k, v, g, beta, s0, cu, 0.1, "kda chunk varlen")
    assert np.array_equal(S[4], s0[4])


@pytest.mark.parametrize("dk,dv,lens", [(64, 64, None), (128, 256, None), (128, 128, [1, 63, 64, 65, 0, 200]),
                                         (64, 128, [1, 63, 64, 65, 0, 200])])
def test_kda_chunk_routes_agree(dk, dv, lens):
    """The workspace route (T and P from the chunk-parallel kernel; at
    d_k = 128 the tensor-core walk over bf16 hi/lo operands) against the
    walk that forms everything itself in fp32, and a repeat of the workspace
    route bitwise."""
    import torch
    if lens is None:
        q, k, v, g, beta, s0, cu = _case(2, 200, 2, dk, dv, seed=31 + dk)
    else:
        q, k, v, g, beta, s0, cu = _case(1, 0, 2, dk, dv, seed=32, seqlens=lens)
    o1, S1 = _run(torch, gdn.gdn_kda_chunk_fwd, q, k, v, g, beta, s0, cu, 0.1)
    o2, S2 = _run(torch, gdn.gdn_kda_chunk_fwd, q, k, v, g, beta, s0, cu, 0.1, tp=True)
    o3, S3 = _run(torch, gdn.gdn_kda_chunk_fwd, q, k, v, g, beta, s0, cu, 0.1, tp=True)
    assert np.array_equal(o2, o3) and np.array_equal(S2, S3)
    G.compare(o2, o1, G.TOL_RMS_IID, G.TOL_MAX_IID, "routes out")
    for s in range(S1.shape[0]):
        G.compare(S2[s], S1[s], TOL_STATE_FP32, None, f"routes state {s}")


@pytest.mark.parametrize("tp", [False, True], ids=["walk", "tp"])
def test_kda_chunk_strong_per_channel_decay(tp):
    """Per-channel log decays down to -40 per token: inside a chunk the
    exponents G_ic - G_jc reach about -2500, far below the fp32 range of exp;
    formed as masked differences they underflow to 0 and never overflow (the
    decayed operands of the tensor-core walk likewise)."""
    import torch
    q, k, v, g, beta, s0, cu = _case(1, 200, 2, 128, 128, seed=13)
    g = (g * 8.0).astype(np.float32)
    scale = 128 ** -0.5
    o, S = _run(torch, gdn.gdn_kda_chunk_fwd, q, k, v, g, beta, s0, cu, scale, tp=tp)
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


# ---------------------------------------------------------------------------
# the chunked backward (gdn_kda_chunk_bwd)
# ---------------------------------------------------------------------------

TOL_DG_FP32 = 1e-3    # dg: fp32 output, a reverse running sum of cancelling terms
TOL_DS0_FP32 = 1e-4   # d_initial_state: fp32 output of the reverse state walk


def _bwd_case(B, T, H, dk, dv, seed, seqlens=None, with_states=True):
    q, k, v, g, beta, s0, cu = _case(B, T, H, dk, dv, seed, seqlens)
    rng = np.random.default_rng(seed + 1000)
    dO = W.f32_to_bf16_bits(rng.standard_normal(v.shape).astype(np.float32))
    dfs = (rng.standard_normal(s0.shape) * 0.1).astype(np.float32) if with_states else None
    return q, k, v, g, beta, (s0 if with_states else None), cu, dO, dfs


def _run_bwd(torch, q, k, v, g, beta, s0, cu, scale, dO, dfs):
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa: E731
    bf = lambda x: d(x.view(np.int16)).view(torch.bfloat16)  # noqa: E731
    r = gdn.chunk_kda_bwd(bf(q), bf(k), bf(v), d(g), bf(beta), bf(dO), scale=scale,
                          initial_state=None if s0 is None else d(s0),
                          cu_seqlens=None if cu is None else d(cu),
                          d_final_state=None if dfs is None else d(dfs))
    st = gdn.gdn_get_last_device_error()
    assert st == 0, gdn.gdn_status_string(st)
    torch.cuda.synchronize()
    res = {n: G.bf16_to_np(r[n]) for n in ("dq", "dk", "dv", "dbeta")}
    res["dg"] = r["dg"].cpu().numpy()
    res["dS0"] = r["d_initial_state"].cpu().numpy()
    return res


def _bounds(q, cu):
    if cu is None:
        return [(b, 0, q.shape[1]) for b in range(q.shape[0])]
    return [(0, int(cu[n]), int(cu[n + 1])) for n in range(len(cu) - 1)]


def _bwd_ref(q, k, v, g, beta, s0, cu, scale, dO, dfs, fn=kda.kda_chunk_bwd_head):
    f = W.bf16_bits_to_f32
    qf, kf, vf, bt, dOf = f(q), f(k), f(v), f(beta), f(dO)
    H = q.shape[2]
    out = dict(dq=np.zeros(q.shape), dk=np.zeros(k.shape), dv=np.zeros(v.shape), dg=np.zeros(g.shape),
               dbeta=np.zeros(beta.shape), dS0=np.zeros((len(_bounds(q, cu)), H, q.shape[3], v.shape[3])))
    for s, (b, t0, t1) in enumerate(_bounds(q, cu)):
        for h in range(H):
            r = fn(qf[b, t0:t1, h], kf[b, t0:t1, h], vf[b, t0:t1, h], g[b, t0:t1, h], bt[b, t0:t1, h], scale,
                   None if s0 is None else s0[s, h], dOf[b, t0:t1, h], None if dfs is None else dfs[s, h])
            for n in ("dq", "dk", "dv", "dg", "dbeta"):
                out[n][b, t0:t1, h] = r[n]
            out["dS0"][s, h] = r["dS0"]
    return out


def _check_bwd(res, ref, q, cu, what, k=None):
    """Per (sequence, head): the bf16 gradients within the gradient tolerance,
    dg and d_initial_state within their fp32 ones.  With k given, dg is
    measured against the size of the terms whose sum it is, q o dq + k o dk,
    instead of its own size: under very strong decay those terms cancel to
    ~1e-9 and only fp32 rounding of the O(1) terms is left (the oracle is
    fp64)."""
    f = W.bf16_bits_to_f32
    for s, (b, t0, t1) in enumerate(_bounds(q, cu)):
        for h in range(q.shape[2]):
            if t1 > t0:
                for n in ("dq", "dk", "dv", "dbeta"):
                    G.compare(res[n][b, t0:t1, h], ref[n][b, t0:t1, h], G.TOL_RMS_GRAD, None,
                              f"{what} {n} s{s} h{h}")
                if k is None:
                    G.compare(res["dg"][b, t0:t1, h], ref["dg"][b, t0:t1, h], TOL_DG_FP32, None,
                              f"{what} dg s{s} h{h}")
                else:
                    terms = (np.abs(f(q[b, t0:t1, h]) * ref["dq"][b, t0:t1, h])
                             + np.abs(f(k[b, t0:t1, h]) * ref["dk"][b, t0:t1, h]))
                    err = np.linalg.norm(res["dg"][b, t0:t1, h] - ref["dg"][b, t0:t1, h]) / np.linalg.norm(terms)
                    assert err <= TOL_DG_FP32, f"{what} dg s{s} h{h}: {err:.3e} of the terms' norm"
            G.compare(res["dS0"][s, h], ref["dS0"][s, h], TOL_DS0_FP32, None, f"{what} dS0 s{s} h{h}")


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128), (128, 256)])
def test_kda_chunk_bwd_matches_oracle(dk, dv):
    """Every gradient against the fp64 reverse mode of the chunk algebra:
    three chunks per sequence with a ragged tail, initial state and an
    upstream gradient on the final state."""
    import torch
    q, k, v, g, beta, s0, cu, dO, dfs = _bwd_case(2, 150, 2, dk, dv, seed=200 + dk + dv)
    scale = dk ** -0.5
    res = _run_bwd(torch, q, k, v, g, beta, s0, cu, scale, dO, dfs)
    _check_bwd(res, _bwd_ref(q, k, v, g, beta, s0, cu, scale, dO, dfs), q, cu, "kda bwd")


def test_kda_chunk_bwd_matches_token_loop_reverse_mode():
    """The same gradients against the reverse mode of the token-by-token
    recurrence (a formulation with no chunk algebra at all)."""
    import torch
    q, k, v, g, beta, s0, cu, dO, dfs = _bwd_case(1, 100, 2, 64, 64, seed=210)
    res = _run_bwd(torch, q, k, v, g, beta, s0, cu, 0.125, dO, dfs)
    ref = _bwd_ref(q, k, v, g, beta, s0, cu, 0.125, dO, dfs, fn=kda.kda_bwd_head)
    _check_bwd(res, ref, q, cu, "kda bwd vs token loop")


def test_kda_chunk_bwd_varlen():
    """Packed sequences of 1, 63, 64, 65, 0 and 130 tokens: the empty one
    hands its final-state gradient to its initial state unchanged."""
    import torch
    lens = [1, 63, 64, 65, 0, 130]
    q, k, v, g, beta, s0, cu, dO, dfs = _bwd_case(1, 0, 2, 128, 64, seed=211, seqlens=lens)
    res = _run_bwd(torch, q, k, v, g, beta, s0, cu, 0.1, dO, dfs)
    _check_bwd(res, _bwd_ref(q, k, v, g, beta, s0, cu, 0.1, dO, dfs), q, cu, "kda bwd varlen")
    assert np.array_equal(res["dS0"][4], dfs[4])


def test_kda_chunk_bwd_without_states_and_exact_chunks():
    """No initial state, no final-state gradient, T a multiple of 64."""
    import torch
    q, k, v, g, beta, s0, cu, dO, dfs = _bwd_case(2, 128, 2, 128, 128, seed=212, with_states=False)
    res = _run_bwd(torch, q, k, v, g, beta, s0, cu, 128 ** -0.5, dO, dfs)
    _check_bwd(res, _bwd_ref(q, k, v, g, beta, s0, cu, 128 ** -0.5, dO, dfs), q, cu, "kda bwd no states")


def test_kda_chunk_bwd_strong_decay_and_repeats_bitwise():
    """Per-channel log decays down to -40 per token stay finite; a second
    call gives the same bits (every sum in a fixed order)."""
    import torch
    q, k, v, g, beta, s0, cu, dO, dfs = _bwd_case(1, 200, 2, 128, 128, seed=213)
    g = (g * 8.0).astype(np.float32)
    r1 = _run_bwd(torch, q, k, v, g, beta, s0, cu, 0.09, dO, dfs)
    r2 = _run_bwd(torch, q, k, v, g, beta, s0, cu, 0.09, dO, dfs)
    for n in r1:
        assert np.isfinite(r1[n]).all(), n
        assert np.array_equal(r1[n], r2[n]), n
    _check_bwd(r1, _bwd_ref(q, k, v, g, beta, s0, cu, 0.09, dO, dfs), q, cu, "kda bwd strong decay", k=k)


def test_kda_chunk_bwd_zero_length():
    import torch
    q, k, v, g, beta, s0, cu, dO, dfs = _bwd_case(2, 0, 2, 64, 64, seed=214)
    res = _run_bwd(torch, q, k, v, g, beta, s0, cu, 0.125, dO, dfs)
    assert np.array_equal(res["dS0"], dfs)


def test_kda_chunk_bwd_long_sequence():
    """T = 4096 (64 chunks through both walks), d_k = d_v = 128."""
    import torch
    q, k, v, g, beta, s0, cu, dO, dfs = _bwd_case(1, 4096, 1, 128, 128, seed=215)
    res = _run_bwd(torch, q, k, v, g, beta, s0, cu, 128 ** -0.5, dO, dfs)
    _check_bwd(res, _bwd_ref(q, k, v, g, beta, s0, cu, 128 ** -0.5, dO, dfs), q, cu, "kda bwd T=4096")


def test_kda_chunk_beta_up_to_two():
    """beta in (0, 2) (the range that allows negative eigenvalues of the
    transition): forward through the workspace route and backward, at
    d_k = 128, against the oracle."""
    import torch
    q, k, v, g, beta, s0, cu, dO, dfs = _bwd_case(2, 150, 2, 128, 128, seed=216)
    beta = W.f32_to_bf16_bits(2.0 * W.bf16_bits_to_f32(beta))
    scale = 128 ** -0.5
    o, S = _run(torch, gdn.gdn_kda_chunk_fwd, q, k, v, g, beta, s0, cu, scale, tp=True)
    _check_against_oracle(o, S, q, k, v, g, beta, s0, cu, scale, "kda beta<2")
    res = _run_bwd(torch, q, k, v, g, beta, s0, cu, scale, dO, dfs)
    _check_bwd(res, _bwd_ref(q, k, v, g, beta, s0, cu, scale, dO, dfs), q, cu, "kda bwd beta<2")
