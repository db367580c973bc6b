"""Failure detection on the GPU without a fault: the forward's issuing warp
first waits, with a short bound, on a hand-off that nothing signals, so the
wait runs out; every CTA records GDN_ERR_TIMEOUT in the device error word and
drains every copy and product it started (with the default bound) before
leaving.  The next call on the same context then runs normally and matches
the oracle."""

import numpy as np
import pytest

from linear_attention_sequence_chunked_gb300 import gdn
from linear_attention_sequence_chunked_gb300 import workloads as W
from oracle import recurrence
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu

GDN_ERR_TIMEOUT = 5


def _forward(wl, d, wait_limit, stall=0):
    import torch
    N, T, H, K, V = wl.n_seq, wl.T, wl.H, wl.d_k, wl.d_v
    out = torch.zeros(d["v"].shape, dtype=torch.bfloat16, device="cuda")
    fs = torch.zeros((N, H, K, V), dtype=torch.float32, device="cuda")
    n = gdn.gdn_chunk_fwd_workspace_size(N, T, H, K, V, wl.cu_seqlens is not None)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    gdn.gdn_chunk_fwd_wait_limit(d["q"], d["k"], d["v"], d["g"], d["beta"], wl.scale, d["initial_state"],
                                 d["cu_seqlens"], out, fs, N, T, H, K, V, ws, n, wait_limit, stall)
    st = gdn.gdn_get_last_device_error()
    return st, out, fs


def test_wait_that_runs_out_reports_timeout_and_the_context_recovers():
    wl = W.random_workload(B=2, T=1024, H=4, d_k=128, d_v=128, seed=31, initial_state=True)
    d = G.to_device(wl)
    for _ in range(2):
        st, _, fs = _forward(wl, d, 64, stall=1)
        assert st == GDN_ERR_TIMEOUT, gdn.gdn_status_string(st)
        # no CTA wrote its final state
        assert not fs.any()
    # the error word was read and cleared; a normal call is correct
    st, out, fs = _forward(wl, d, 0)
    assert st == 0, gdn.gdn_status_string(st)
    o_ref, S_ref = recurrence.workload_fwd(wl)
    G.compare(G.bf16_to_np(out), o_ref, G.TOL_RMS_IID, G.TOL_MAX_IID, "after timeout: out")
    G.compare(fs.cpu().numpy(), S_ref, G.TOL_RMS_IID, G.TOL_MAX_IID, "after timeout: state")


def test_default_bound_through_the_wait_limit_entry_is_gdn_chunk_fwd():
    wl = W.random_workload(B=1, T=300, H=2, d_k=128, d_v=64, seed=32, initial_state=True)
    d = G.to_device(wl)
    st, out, fs = _forward(wl, d, 0)
    assert st == 0
    o, S = G.run_fwd(wl)
    assert np.array_equal(G.bf16_to_np(out), o) and np.array_equal(fs.cpu().numpy(), S)
