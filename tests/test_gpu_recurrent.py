"""The token-serial forward (gdn_recurrent_fwd): parity with the fp64 oracle,
agreement with the chunked forward, and decode one token per call."""

import numpy as np
import pytest

from linear_attention_sequence_chunked_gb300 import gdn
from linear_attention_sequence_chunked_gb300 import workloads as W
from oracle import recurrence
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu


def run_recurrent(wl, initial_state=None, dev="cuda"):
    import torch
    d = G.to_device(wl, dev)
    n_seq = wl.n_seq
    out = torch.empty(d["v"].shape, dtype=torch.bfloat16, device=dev)
    fs = torch.empty((n_seq, wl.H, wl.d_k, wl.d_v), dtype=torch.float32, device=dev)
    s0 = d["initial_state"] if initial_state is None else initial_state
    B = n_seq if wl.cu_seqlens is not None else wl.B
    gdn.gdn_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], wl.scale, s0,
                          d["cu_seqlens"], out, fs, B, wl.T, wl.H, wl.d_k, wl.d_v)
    st = gdn.gdn_get_last_device_error()
    assert st == 0, gdn.gdn_status_string(st)
    torch.cuda.synchronize()
    return G.bf16_to_np(out), fs.cpu().numpy(), fs


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 256), (128, 128)])
@pytest.mark.parametrize("T", [1, 65, 300])
def test_recurrent_matches_oracle(T, dk, dv):
    wl = W.random_workload(B=2, T=T, H=2, d_k=dk, d_v=dv, seed=T + dk, initial_state=True)
    o, S, _ = run_recurrent(wl)
    o_ref, S_ref = recurrence.workload_fwd(wl)
    G.compare(o, o_ref, G.TOL_RMS_IID, G.TOL_MAX_IID, f"T={T} out")
    G.compare(S, S_ref, 1e-5, None, f"T={T} state")


def test_recurrent_varlen():
    lens = [1, 63, 0, 200, 64]
    wl = W.random_workload(B=1, T=0, H=3, d_k=128, d_v=128, seed=21, seqlens=lens,
                           initial_state=True)
    o, S, _ = run_recurrent(wl)
    o_ref, S_ref = recurrence.workload_fwd(wl)
    G.compare(o, o_ref, G.TOL_RMS_IID, G.TOL_MAX_IID, "varlen out")
    for s in range(len(lens)):
        G.compare(S[s], S_ref[s], 1e-5, None, f"varlen state {s}")
    assert np.array_equal(S[2], wl.initial_state[2])


def test_recurrent_agrees_with_chunked_forward():
    """Two independent GPU paths (token-serial fp32, chunked tensor-core)."""
    wl = W.make_workload(2, B=2, H=4, T=1024)
    o_r, S_r, _ = run_recurrent(wl)
    o_c, S_c = G.run_fwd(wl)
    G.compare(o_c, o_r, 3e-3, 1e-2, "chunked vs recurrent out")
    G.compare(S_c, S_r, 1e-4, None, "chunked vs recurrent state")


def test_decode_one_token_per_call_is_bitwise_equal():
    """Decoding token by token (state carried through final_state ->
    initial_state) gives the same bits as one call over the sequence."""
    import torch
    wl = W.random_workload(B=1, T=40, H=2, d_k=128, d_v=64, seed=8, initial_state=True)
    o_all, S_all, _ = run_recurrent(wl)
    state = torch.from_numpy(wl.initial_state).to("cuda")
    outs = []
    for t in range(wl.T):
        step = W.Workload(name="step", q=np.ascontiguousarray(wl.q[:, t:t + 1]),
                          k=np.ascontiguousarray(wl.k[:, t:t + 1]),
                          v=np.ascontiguousarray(wl.v[:, t:t + 1]),
                          g=np.ascontiguousarray(wl.g[:, t:t + 1]),
                          beta=np.ascontiguousarray(wl.beta[:, t:t + 1]), scale=wl.scale,
                          initial_state=wl.initial_state)
        o1, _, fs = run_recurrent(step, initial_state=state)
        state = fs.clone()
        outs.append(o1)
    assert np.array_equal(np.concatenate(outs, axis=1), o_all)
    assert np.array_equal(state.cpu().numpy(), S_all)
