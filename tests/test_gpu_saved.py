"""The training route: gdn_chunk_fwd_save keeps every chunk's start state and
T tiles, gdn_chunk_bwd_saved reuses them.  Outputs and gradients are bitwise
those of the recomputing route (gdn_chunk_fwd, gdn_chunk_bwd) and match the
fp64 oracle; the backward launches only its last two passes and leaves the
saved buffer as it found it."""

import numpy as np
import pytest

from linear_attention_sequence_chunked_gb300 import gdn
from linear_attention_sequence_chunked_gb300 import workloads as W
from oracle import recurrence
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu

GRADS = ("dq", "dk", "dv", "dg", "dbeta", "d_initial_state")


def _routes(wl):
    import torch
    d = G.to_device(wl)
    common = dict(scale=wl.scale, initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"])
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"])
    out_a, fs_a = gdn.chunk_gated_delta_rule_fwd(*args, **common)
    ra = gdn.chunk_gated_delta_rule_bwd(*args, d["d_out"], d_final_state=d["d_final_state"], **common)
    n0 = gdn.gdn_kernel_launches()
    out_b, fs_b, saved = gdn.chunk_gated_delta_rule_fwd(*args, save_for_backward=True, **common)
    n1 = gdn.gdn_kernel_launches()
    torch.cuda.synchronize()
    snapshot = saved.clone()
    rb = gdn.chunk_gated_delta_rule_bwd(*args, d["d_out"], d_final_state=d["d_final_state"], saved=saved,
                                        **common)
    n2 = gdn.gdn_kernel_launches()
    st = gdn.gdn_get_last_device_error()
    assert st == 0, gdn.gdn_status_string(st)
    torch.cuda.synchronize()
    assert torch.equal(saved, snapshot), "the saved buffer changed"
    return (out_a, fs_a, ra), (out_b, fs_b, rb), (n1 - n0, n2 - n1)


def _bits(t):
    import torch
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def _assert_bitwise(a, b):
    import torch
    (out_a, fs_a, ra), (out_b, fs_b, rb) = a, b
    assert torch.equal(_bits(out_a), _bits(out_b)), "out"
    assert torch.equal(_bits(fs_a), _bits(fs_b)), "final state"
    for n in GRADS:
        assert torch.equal(_bits(ra[n]), _bits(rb[n])), n


CASES = [
    dict(B=2, T=300, H=3, d_k=128, d_v=128),
    dict(B=2, T=200, H=2, d_k=64, d_v=64),
    dict(B=1, T=130, H=2, d_k=128, d_v=256),
    dict(B=2, T=64, H=1, d_k=64, d_v=128),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{B}T{T}H{H}k{d_k}v{d_v}".format(**c))
def test_saved_route_is_bitwise_the_recomputing_route(case):
    wl = W.random_workload(**case, seed=case["T"] + case["d_v"], beta_max=2.0, initial_state=True,
                           with_grad=True, d_final_state=True)
    a, b, (n_fwd, n_bwd) = _routes(wl)
    _assert_bitwise(a, b)
    assert n_fwd == 2 and n_bwd == 2   # T kernel + chain;  reverse chain + gradient pass
    # and against the oracle
    out_b, fs_b, rb = b
    o_ref, s_ref = recurrence.workload_fwd(wl)
    G.compare(G.bf16_to_np(out_b), o_ref, G.TOL_RMS_IID, G.TOL_MAX_IID, "out")
    G.compare(fs_b.cpu().numpy(), s_ref, G.TOL_RMS_IID, G.TOL_MAX_IID, "final state")
    ref = recurrence.workload_bwd(wl)
    for n in ("dq", "dk", "dv", "dbeta"):
        G.compare(G.bf16_to_np(rb[n]), ref[n], G.TOL_RMS_GRAD, None, n)
    G.compare(rb["dg"].cpu().numpy(), ref["dg"], G.TOL_RMS_GRAD, None, "dg")
    G.compare(rb["d_initial_state"].cpu().numpy(), ref["dS0"], G.TOL_RMS_GRAD, None, "dS0")


def test_saved_route_packed_sequences():
    lens = [1, 63, 65, 0, 700, 64, 129]
    wl = W.random_workload(B=1, T=0, H=2, d_k=128, d_v=128, seed=23, seqlens=lens, initial_state=True,
                           with_grad=True, d_final_state=True)
    a, b, _ = _routes(wl)
    _assert_bitwise(a, b)
    rb = b[2]
    units = [(s, h) for s in range(len(lens)) for h in range(2)]
    ref = recurrence.workload_bwd(wl, units=units)
    for (bb, t0, t1, h, s) in G.unit_rows(wl, units):
        if t1 > t0:
            G.compare(G.bf16_to_np(rb["dk"])[bb, t0:t1, h], ref["dk"][bb, t0:t1, h], G.TOL_RMS_GRAD, None,
                      f"dk s{s} h{h}")
        G.compare(rb["d_initial_state"].cpu().numpy()[s, h], ref["dS0"][s, h], G.TOL_RMS_GRAD, None,
                  f"dS0 s{s} h{h}")


def test_saved_route_zero_length():
    import torch
    wl = W.random_workload(B=2, T=0, H=2, d_k=64, d_v=64, seed=3, initial_state=True, with_grad=True,
                           d_final_state=True)
    a, b, _ = _routes(wl)
    _assert_bitwise(a, b)
    # nothing to save, and the state gradient passes straight through
    assert gdn.gdn_chunk_saved_size(2, 0, 2, 64, 64, 0) == 0
    assert torch.equal(b[2]["d_initial_state"].cpu(), torch.from_numpy(wl.d_final_state))


def test_saved_route_full_size_matches_recomputing_route():
    """B=4, H=16, T=4096, d_k=d_v=128, the configuration the benchmark times:
    the two routes agree bit for bit, and sampled heads match the oracle."""
    wl = W.make_workload(2, with_grad=True)
    a, b, _ = _routes(wl)
    _assert_bitwise(a, b)
    units = [(0, 0), (3, 15)]
    ref = recurrence.workload_bwd(wl, units=units)
    rb = b[2]
    for (bb, t0, t1, h, s) in G.unit_rows(wl, units):
        for n in ("dq", "dk", "dv"):
            G.compare(G.bf16_to_np(rb[n])[bb, t0:t1, h], ref[n][bb, t0:t1, h], G.TOL_RMS_GRAD, None,
                      f"{n} s{s} h{h}")
    assert np.isfinite(G.bf16_to_np(b[0])).all()


@pytest.mark.parametrize("dk,dv", [(64, 256), (64, 64)])
def test_saved_route_packed_other_widths(dk, dv):
    """Packed sequences at the other key and value widths: the training route
    stays bitwise the recomputing route."""
    lens = [70, 0, 129, 64, 1]
    wl = W.random_workload(B=1, T=0, H=2, d_k=dk, d_v=dv, seed=dk + dv, seqlens=lens, initial_state=True,
                           with_grad=True, d_final_state=True, beta_max=2.0)
    a, b, (n_fwd, n_bwd) = _routes(wl)
    _assert_bitwise(a, b)
    assert n_fwd == 2 and n_bwd == 2
