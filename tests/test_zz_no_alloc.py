"""The backward entry point that allocates nothing (gdn_chunk_bwd_noalloc).

Some callers may not allocate device memory themselves -- a runtime that
fixes its memory plan at start-up, or a plugin whose host framework owns all
device allocations -- so they cannot pass the workspace gdn_chunk_bwd needs.
gdn_chunk_bwd_noalloc takes its scratch from an array built into the library
instead.  This file is collected last on purpose: it checks the variant
against the ordinary entry point, twice in a row (the shared scratch keeps
the previous call's contents), and it passes alone or after the other tests.
"""

import numpy as np
import pytest

from linear_attention_sequence_chunked_gb300 import gdn
from linear_attention_sequence_chunked_gb300 import workloads as W
from oracle import metrics, recurrence
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu


def _noalloc_bwd(wl):
    import torch
    d = G.to_device(wl)
    B = wl.n_seq
    dev = "cuda"
    out = dict(dq=torch.empty(d["q"].shape, dtype=torch.bfloat16, device=dev),
               dk=torch.empty(d["k"].shape, dtype=torch.bfloat16, device=dev),
               dv=torch.empty(d["v"].shape, dtype=torch.bfloat16, device=dev),
               dg=torch.empty(d["g"].shape, dtype=torch.float32, device=dev),
               dbeta=torch.empty(d["beta"].shape, dtype=torch.bfloat16, device=dev),
               dS0=torch.empty((B, wl.H, wl.d_k, wl.d_v), dtype=torch.float32, device=dev))
    gdn.gdn_chunk_bwd_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], wl.scale,
                              d["initial_state"], d["cu_seqlens"], d["d_out"], d["d_final_state"],
                              out["dq"], out["dk"], out["dv"], out["dg"], out["dbeta"], out["dS0"],
                              B, wl.T, wl.H, wl.d_k, wl.d_v)
    assert gdn.gdn_get_last_device_error() == 0
    res = {n: G.bf16_to_np(out[n]) for n in ("dq", "dk", "dv", "dbeta")}
    res["dg"] = out["dg"].cpu().numpy()
    res["dS0"] = out["dS0"].cpu().numpy()
    return res


def test_noalloc_backward_matches_workspace_backward_twice():
    """Same kernels on the same values as gdn_chunk_bwd with a caller
    workspace, so every gradient must be bitwise equal, on the first call and
    on a second one that finds the previous call's scratch contents; both
    also within the gradient tolerance of the fp64 reverse-mode oracle."""
    wl = W.random_workload(B=2, T=200, H=2, d_k=128, d_v=128, seed=21, beta_max=2.0,
                           initial_state=True, with_grad=True, d_final_state=True)
    ref = G.run_bwd(wl)
    units = [(s, h) for s in range(2) for h in range(2)]
    oracle = recurrence.workload_bwd(wl, units=units)
    for call in range(2):
        res = _noalloc_bwd(wl)
        for name in ref:
            assert np.all(np.isfinite(res[name])), (call, name)
            assert np.array_equal(res[name].view(np.uint32), ref[name].view(np.uint32)), (call, name)
        for (b, t0, t1, h, s) in G.unit_rows(wl, units):
            for name in ("dq", "dk", "dv", "dg", "dbeta"):
                e = metrics.rel_l2(res[name][b, t0:t1, h], oracle[name][b, t0:t1, h])
                assert e <= G.TOL_RMS_GRAD, (call, name, s, h, e)
            e = metrics.rel_l2(res["dS0"][s, h], oracle["dS0"][s, h])
            assert e <= G.TOL_RMS_GRAD, (call, "dS0", s, h, e)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import torch
    # B=8, T=4096, H=16, d=128 needs far more than the built-in scratch
    need = gdn.gdn_chunk_bwd_workspace_size(8, 4096, 16, 128, 128, 0)
    assert need > (64 << 20)
    x = torch.empty(16, dtype=torch.bfloat16, device="cuda")  # never read: rejected first
    with pytest.raises(gdn.GdnError) as err:
        gdn.gdn_chunk_bwd_noalloc(x, x, x, x, x, 1.0, None, None, x, None, x, x, x, x, x, None,
                                  8, 4096, 16, 128, 128)
    assert err.value.status == 2
