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


def _backward_saved(wl, d, wait_limit, stall=0):
    """The training route's backward (gradient pass through the wait-limit
    entry) on the saving forward's buffer; gradients start as zeros."""
    import torch
    N, T, H, K, V = wl.n_seq, wl.T, wl.H, wl.d_k, wl.d_v
    varlen = wl.cu_seqlens is not None
    out = torch.empty(d["v"].shape, dtype=torch.bfloat16, device="cuda")
    fs = torch.empty((N, H, K, V), dtype=torch.float32, device="cuda")
    ns = gdn.gdn_chunk_saved_size(N, T, H, K, V, varlen)
    saved = torch.empty(ns, dtype=torch.uint8, device="cuda")
    gdn.gdn_chunk_fwd_save(d["q"], d["k"], d["v"], d["g"], d["beta"], wl.scale, d["initial_state"],
                           d["cu_seqlens"], out, fs, N, T, H, K, V, saved, ns)
    nb = gdn.gdn_chunk_bwd_saved_workspace_size(N, T, H, K, V, varlen)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    r = dict(dq=torch.zeros_like(d["q"]), dk=torch.zeros_like(d["k"]), dv=torch.zeros_like(d["v"]),
             dg=torch.zeros_like(d["g"]), dbeta=torch.zeros_like(d["beta"]),
             dS0=torch.zeros((N, H, K, V), dtype=torch.float32, device="cuda"))
    gdn.gdn_chunk_bwd_saved_wait_limit(d["q"], d["k"], d["v"], d["g"], d["beta"], wl.scale, d["cu_seqlens"],
                                       d["d_out"], d["d_final_state"], r["dq"], r["dk"], r["dv"], r["dg"],
                                       r["dbeta"], r["dS0"], N, T, H, K, V, saved, ns, ws, nb,
                                       wait_limit, stall)
    st = gdn.gdn_get_last_device_error()
    return st, r


def test_gradient_pass_wait_that_runs_out_reports_timeout_and_the_context_recovers():
    """The chunk-parallel gradient pass (epilogue warps + MMA-issuing warp):
    its epilogue warps first wait on a barrier that nothing signals; at the
    next hand-off the issuing warp leaves with them, no gradient is written,
    and the next call is bitwise the ordinary entry point's."""
    wl = W.random_workload(B=2, T=1024, H=4, d_k=128, d_v=128, seed=33, initial_state=True,
                           with_grad=True, d_final_state=True)
    d = G.to_device(wl)
    for _ in range(2):
        st, r = _backward_saved(wl, d, 64, stall=1)
        assert st == GDN_ERR_TIMEOUT, gdn.gdn_status_string(st)
        for name in ("dq", "dk", "dv", "dg", "dbeta"):
            assert not r[name].any(), name
    st, r = _backward_saved(wl, d, 0)
    assert st == 0, gdn.gdn_status_string(st)
    res = G.run_bwd(wl)
    for name in ("dq", "dk", "dv", "dbeta"):
        assert np.array_equal(G.bf16_to_np(r[name]), res[name]), name
    assert np.array_equal(r["dg"].cpu().numpy(), res["dg"])
    assert np.array_equal(r["dS0"].cpu().numpy(), res["dS0"])
