"""Edge cases, index-exact varlen resets, resume, determinism and the device
error word."""

import numpy as np
import pytest

from linear_attention_sequence_chunked_gb300 import gdn
from linear_attention_sequence_chunked_gb300 import workloads as W
from oracle import recurrence
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [1, 63, 64, 65, 129])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 256)])
def test_short_and_ragged_lengths(T, dk, dv):
    wl = W.random_workload(B=2, T=T, H=2, d_k=dk, d_v=dv, seed=T, initial_state=True)
    o, S = G.run_fwd(wl)
    units = [(s, h) for s in range(2) for h in range(2)]
    o_ref, S_ref = recurrence.workload_fwd(wl, units=units)
    G.compare(o, o_ref, G.TOL_RMS_IID, G.TOL_MAX_IID, f"T={T} out")
    G.compare(S, S_ref, G.TOL_RMS_IID, G.TOL_MAX_IID, f"T={T} state")


def test_varlen_matches_oracle_with_empty_and_tiny_sequences():
    lens = [1, 63, 65, 0, 5120, 64]
    wl = W.random_workload(B=1, T=0, H=3, d_k=128, d_v=128, seed=3, seqlens=lens,
                           initial_state=True)
    o, S = G.run_fwd(wl)
    o_ref, S_ref = recurrence.workload_fwd(wl)
    G.compare(o, o_ref, G.TOL_RMS_IID, G.TOL_MAX_IID, "varlen out")
    for s in range(len(lens)):
        G.compare(S[s], S_ref[s], G.TOL_RMS_IID, G.TOL_MAX_IID, f"varlen state {s}")
    # the empty sequence hands its initial state through unchanged
    assert np.array_equal(S[3], wl.initial_state[3])


def test_varlen_is_index_exact_against_separate_calls():
    """A packed call equals one call per sequence, bit for bit."""
    lens = [100, 1, 257, 64]
    wl = W.random_workload(B=1, T=0, H=2, d_k=64, d_v=128, seed=9, seqlens=lens,
                           initial_state=True)
    o, S = G.run_fwd(wl)
    for s, (b, t0, t1) in enumerate(wl.seq_bounds()):
        single = W.Workload(name="one", q=wl.q[:, t0:t1], k=wl.k[:, t0:t1], v=wl.v[:, t0:t1],
                            g=np.ascontiguousarray(wl.g[:, t0:t1]),
                            beta=np.ascontiguousarray(wl.beta[:, t0:t1]), scale=wl.scale,
                            initial_state=np.ascontiguousarray(wl.initial_state[s:s + 1]))
        single.q = np.ascontiguousarray(single.q)
        single.k = np.ascontiguousarray(single.k)
        single.v = np.ascontiguousarray(single.v)
        o1, S1 = G.run_fwd(single)
        assert np.array_equal(o1[0], o[0, t0:t1]), s
        assert np.array_equal(S1[0], S[s]), s


def test_resume_from_final_state():
    """fwd(T1) then fwd(T2) from its final state equals fwd(T1 + T2): bitwise
    when T1 is a multiple of the chunk, within tolerance otherwise."""
    wl = W.random_workload(B=1, T=300, H=2, d_k=128, d_v=64, seed=4, initial_state=True)
    o, S = G.run_fwd(wl)
    for T1, exact in [(128, True), (100, False)]:
        a = W.Workload(name="a", q=np.ascontiguousarray(wl.q[:, :T1]),
                       k=np.ascontiguousarray(wl.k[:, :T1]), v=np.ascontiguousarray(wl.v[:, :T1]),
                       g=np.ascontiguousarray(wl.g[:, :T1]),
                       beta=np.ascontiguousarray(wl.beta[:, :T1]), scale=wl.scale,
                       initial_state=wl.initial_state)
        oa, Sa = G.run_fwd(a)
        b = W.Workload(name="b", q=np.ascontiguousarray(wl.q[:, T1:]),
                       k=np.ascontiguousarray(wl.k[:, T1:]), v=np.ascontiguousarray(wl.v[:, T1:]),
                       g=np.ascontiguousarray(wl.g[:, T1:]),
                       beta=np.ascontiguousarray(wl.beta[:, T1:]), scale=wl.scale,
                       initial_state=Sa)
        ob, Sb = G.run_fwd(b)
        if exact:
            assert np.array_equal(np.concatenate([oa, ob], axis=1), o)
            assert np.array_equal(Sb, S)
        else:
            G.compare(np.concatenate([oa, ob], axis=1), o, 1e-3, None, "resume out")
            G.compare(Sb, S, 1e-4, None, "resume state")


@pytest.mark.parametrize("dk,dv,lens", [(128, 128, [1, 63, 65, 0, 700, 64]), (64, 256, [129, 300])])
def test_forward_routes_agree_bitwise(dk, dv, lens):
    """T from the chunk-parallel kernel (workspace given) and T formed inside
    the chunk chain (no workspace) give the same bits; both routes also match
    the oracle."""
    import torch
    wl = W.random_workload(B=1, T=0, H=2, d_k=dk, d_v=dv, seed=11, seqlens=lens,
                           initial_state=True)
    d = G.to_device(wl)
    N = len(lens)
    outs = []
    for with_ws in (True, False):
        out = torch.empty(d["v"].shape, dtype=torch.bfloat16, device="cuda")
        fs = torch.empty((N, 2, dk, dv), dtype=torch.float32, device="cuda")
        nbytes = gdn.gdn_chunk_fwd_workspace_size(N, wl.T, 2, dk, dv, True)
        assert nbytes > 0
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda") if with_ws else None
        gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], wl.scale,
                          d["initial_state"], d["cu_seqlens"], out, fs, N, wl.T, 2, dk, dv,
                          ws, nbytes if with_ws else 0)
        assert gdn.gdn_get_last_device_error() == 0
        torch.cuda.synchronize()
        outs.append((G.bf16_to_np(out), fs.cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0])
    assert np.array_equal(outs[0][1], outs[1][1])
    o_ref, S_ref = recurrence.workload_fwd(wl)
    for r, name in ((0, "workspace"), (1, "no-workspace")):
        G.compare(outs[r][0], o_ref, G.TOL_RMS_IID, G.TOL_MAX_IID, f"{name} out")
        G.compare(outs[r][1], S_ref, G.TOL_RMS_IID, G.TOL_MAX_IID, f"{name} state")


def test_repeat_launches_are_bitwise_equal():
    wl = W.make_workload(2, B=2, H=4, T=1024, with_grad=True)
    o1, S1 = G.run_fwd(wl)
    o2, S2 = G.run_fwd(wl)
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)
    g1 = G.run_bwd(wl)
    g2 = G.run_bwd(wl)
    for n in g1:
        assert np.array_equal(g1[n], g2[n]), n


def test_zero_length_passes_state_through():
    import torch
    wl = W.random_workload(B=2, T=0, H=2, d_k=64, d_v=64, seed=1, initial_state=True)
    o, S = G.run_fwd(wl)
    assert o.size == 0
    assert np.array_equal(S, wl.initial_state)
    torch.cuda.synchronize()


def test_bad_cu_seqlens_sets_device_error_and_writes_nothing():
    import torch
    wl = W.random_workload(B=1, T=0, H=2, d_k=64, d_v=64, seed=2, seqlens=[64, 64])
    d = G.to_device(wl)
    for bad in ([0, 100, 64], [0, 64, 120], [3, 64, 128]):
        cu = torch.tensor(bad, dtype=torch.int32, device="cuda")
        out = torch.full(d["v"].shape, 7.0, dtype=torch.bfloat16, device="cuda")
        fs = torch.full((2, 2, 64, 64), 5.0, dtype=torch.float32, device="cuda")
        gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], wl.scale, None, cu, out, fs,
                          2, wl.T, 2, 64, 64)
        st = gdn.gdn_get_last_device_error()
        assert st == 4, gdn.gdn_status_string(st)
        assert gdn.gdn_get_last_device_error() == 0  # cleared
    # a good call afterwards still works
    o, S = G.run_fwd(wl)
    assert np.all(np.isfinite(o))
