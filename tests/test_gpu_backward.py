"""GPU backward parity against the fp64 reverse-mode oracle."""

import pytest

from linear_attention_sequence_chunked_gb300 import workloads as W
from oracle import recurrence
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dg", "dbeta")


def _check_grads(wl, res, units, tag):
    ref = recurrence.workload_bwd(wl, units=units)
    for (b, t0, t1, h, s) in G.unit_rows(wl, units):
        for n in NAMES:
            G.compare(res[n][b, t0:t1, h], ref[n][b, t0:t1, h], G.TOL_RMS_GRAD, None,
                      f"{tag} {n} s{s} h{h}")
        G.compare(res["dS0"][s, h], ref["dS0"][s, h], G.TOL_RMS_GRAD, None, f"{tag} dS0 s{s} h{h}")


def test_config5_training_heads():
    """B=8, T=4096, H=16, d_k=128, d_v=256, beta in (0,2): gradients of heads
    0 and 15 of batch 0 against the reverse-mode oracle."""
    wl = W.make_workload(5, with_grad=True)
    res = G.run_bwd(wl)
    _check_grads(wl, res, [(0, 0), (0, 15)], "cfg5")


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 128), (128, 256)])
def test_small_all_heads(dk, dv):
    wl = W.random_workload(B=2, T=200, H=2, d_k=dk, d_v=dv, seed=dk + dv, beta_max=2.0,
                           initial_state=True, with_grad=True, d_final_state=True)
    res = G.run_bwd(wl)
    _check_grads(wl, res, [(s, h) for s in range(2) for h in range(2)], f"small {dk}x{dv}")


def test_varlen_gradients():
    wl = W.random_workload(B=1, T=0, H=2, d_k=64, d_v=64, seed=5, seqlens=[1, 63, 65, 130, 0, 64],
                           initial_state=True, with_grad=True, d_final_state=True)
    res = G.run_bwd(wl)
    _check_grads(wl, res, [(s, h) for s in range(wl.n_seq) for h in range(2) if s != 4], "varlen")
    ref = recurrence.workload_bwd(wl, units=[(4, 0), (4, 1)])
    # an empty sequence passes the final-state gradient straight through
    for h in range(2):
        G.compare(res["dS0"][4, h], ref["dS0"][4, h], 1e-6, None, "empty seq")


def test_varlen_gradients_dk128_many_items():
    """Packed sequences at d_k=128 with more (chunk, head) items than SMs: the
    persistent local-gradient pass walks several items per CTA, including
    ragged tails read by TMA and empty or one-token sequences."""
    lens = [1, 63, 65, 0, 3000, 64, 129, 700]
    wl = W.random_workload(B=1, T=0, H=3, d_k=128, d_v=128, seed=17, seqlens=lens,
                           initial_state=True, with_grad=True, d_final_state=True)
    res = G.run_bwd(wl)
    _check_grads(wl, res, [(s, h) for s in range(len(lens)) for h in range(3) if lens[s] > 0],
                 "varlen128")


def test_config2_shape_gradients_sampled():
    wl = W.make_workload(2, with_grad=True)
    res = G.run_bwd(wl)
    _check_grads(wl, res, [(0, 0), (3, 15)], "cfg2")
