"""chunk_gated_delta_rule under torch.autograd: the gradients are bitwise
those of the explicit training route and match the fp64 oracle."""

import pytest

from linear_attention_sequence_chunked_gb300 import gdn
from linear_attention_sequence_chunked_gb300 import workloads as W
from oracle import recurrence
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("packed", [False, True])
def test_autograd_gradients(packed):
    import torch
    if packed:
        wl = W.random_workload(B=1, T=0, H=2, d_k=128, d_v=128, seed=31, seqlens=[70, 129, 1],
                               initial_state=True, with_grad=True, d_final_state=True, beta_max=2.0)
    else:
        wl = W.random_workload(B=2, T=200, H=2, d_k=128, d_v=64, seed=32, initial_state=True,
                               with_grad=True, d_final_state=True, beta_max=2.0)
    d = G.to_device(wl)
    leaves = {n: d[n].clone().requires_grad_(True) for n in ("q", "k", "v", "g", "beta", "initial_state")}
    out, fs = gdn.chunk_gated_delta_rule(leaves["q"], leaves["k"], leaves["v"], leaves["g"], leaves["beta"],
                                         scale=wl.scale, initial_state=leaves["initial_state"],
                                         cu_seqlens=d["cu_seqlens"])
    torch.autograd.backward([out, fs], [d["d_out"], d["d_final_state"]])
    torch.cuda.synchronize()
    # the explicit route on the same inputs
    _, _, res = G.run_train(wl)
    names = {"q": "dq", "k": "dk", "v": "dv", "beta": "dbeta", "g": "dg", "initial_state": "dS0"}
    for leaf, n in names.items():
        grad = leaves[leaf].grad
        got = G.bf16_to_np(grad) if grad.dtype == torch.bfloat16 else grad.cpu().numpy()
        assert (got == res[n]).all(), leaf
    ref = recurrence.workload_bwd(wl)
    G.compare(G.bf16_to_np(leaves["k"].grad), ref["dk"], G.TOL_RMS_GRAD, None, "dk")
    G.compare(leaves["initial_state"].grad.cpu().numpy(), ref["dS0"], G.TOL_RMS_GRAD, None, "dS0")
