"""The prologue (q/k L2 normalisation, gates) and its reverse mode against the
fp64 prologue oracle, and end to end through the chunked operator."""

import math

import numpy as np
import pytest

from linear_attention_sequence_chunked_gb300 import gdn
from linear_attention_sequence_chunked_gb300 import workloads as W
from oracle import metrics
from oracle import prologue as P
from oracle import recurrence
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu

MODES = [(1, -5.0, 1.0), (1, -5.0, 2.0), (2, -5.0, 1.0)]


def _dev_bf16(x, torch):
    return torch.from_numpy(W.f32_to_bf16_bits(np.asarray(x, np.float32)).view(np.int16)).cuda().view(
        torch.bfloat16)


def _f32(x):
    """bf16 bits of float32 values, back to float32 (what the device holds)."""
    return W.bf16_bits_to_f32(W.f32_to_bf16_bits(np.asarray(x, np.float32)))


def _inputs(rows, H, dk, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((rows, H, dk)).astype(np.float32) * 3
    k = rng.standard_normal((rows, H, dk)).astype(np.float32) * 0.5
    q[3, 1] = 0.0  # a zero row maps to zero
    a = rng.standard_normal((rows, H)).astype(np.float32) * 2
    b = rng.standard_normal((rows, H)).astype(np.float32) * 2
    A_log = rng.uniform(0, math.log(16), H).astype(np.float32)
    dtb = rng.uniform(-1, 1, H).astype(np.float32)
    return _f32(q), _f32(k), a, b, A_log, dtb


def _run_fwd(torch, q, k, a, b, A_log, dtb, mode, lower, bs):
    rows, H, dk = q.shape
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa: E731
    qo = torch.empty((rows, H, dk), dtype=torch.bfloat16, device="cuda")
    ko = torch.empty_like(qo)
    go = torch.empty((rows, H), dtype=torch.float32, device="cuda")
    bo = torch.empty((rows, H), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_prologue_fwd(_dev_bf16(q, torch), _dev_bf16(k, torch), t(a), t(b),
                         t(A_log) if mode == 1 else None, t(dtb), mode, lower, bs, qo, ko, go, bo,
                         rows, H, dk)
    torch.cuda.synchronize()
    return qo, ko, go, bo


@pytest.mark.parametrize("dk", [64, 128])
@pytest.mark.parametrize("mode,lower,bs", MODES)
def test_prologue_forward_matches_oracle(dk, mode, lower, bs):
    import torch
    q, k, a, b, A_log, dtb = _inputs(300, 4, dk, seed=dk + mode)
    qo, ko, go, bo = _run_fwd(torch, q, k, a, b, A_log, dtb, mode, lower, bs)
    qh, kh = P.l2norm(q), P.l2norm(k)
    g_ref, b_ref = P.gates(a, b, A_log, dtb, mode="decay" if mode == 1 else "bounded", lower=lower,
                           beta_scale=bs)
    G.compare(G.bf16_to_np(qo), qh, G.TOL_RMS_IID, G.TOL_MAX_IID, "q_hat")
    G.compare(G.bf16_to_np(ko), kh, G.TOL_RMS_IID, G.TOL_MAX_IID, "k_hat")
    assert np.all(G.bf16_to_np(qo)[3, 1] == 0.0)
    G.compare(go.cpu().numpy(), g_ref, 1e-5, 1e-5, "g")
    G.compare(G.bf16_to_np(bo), b_ref, G.TOL_RMS_IID, G.TOL_MAX_IID, "beta")


@pytest.mark.parametrize("mode,lower,bs", MODES)
def test_prologue_backward_matches_oracle(mode, lower, bs):
    import torch
    rows, H, dk = 257, 3, 128
    q, k, a, b, A_log, dtb = _inputs(rows, H, dk, seed=40 + mode)
    rng = np.random.default_rng(7)
    dq = _f32(rng.standard_normal((rows, H, dk)))
    dk_ = _f32(rng.standard_normal((rows, H, dk)))
    dg = rng.standard_normal((rows, H)).astype(np.float32)
    dbeta = _f32(rng.standard_normal((rows, H)))
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa: E731
    out = {n: torch.empty((rows, H, dk), dtype=torch.bfloat16, device="cuda") for n in ("dq", "dk")}
    da = torch.empty((rows, H), dtype=torch.float32, device="cuda")
    db = torch.empty_like(da)
    dA = torch.empty((H,), dtype=torch.float32, device="cuda")
    ddt = torch.empty_like(dA)
    gdn.gdn_prologue_bwd(_dev_bf16(q, torch), _dev_bf16(k, torch), t(a), t(b),
                         t(A_log) if mode == 1 else None, t(dtb), mode, lower, bs,
                         _dev_bf16(dq, torch), _dev_bf16(dk_, torch), t(dg), _dev_bf16(dbeta, torch),
                         out["dq"], out["dk"], da, db, dA if mode == 1 else None, ddt, rows, H, dk)
    torch.cuda.synchronize()
    m = "decay" if mode == 1 else "bounded"
    da_r, db_r, dA_r, ddt_r = P.gates_bwd(a, b, dg, dbeta, A_log, dtb, mode=m, lower=lower, beta_scale=bs)
    G.compare(G.bf16_to_np(out["dq"]), P.l2norm_bwd(q, dq), G.TOL_RMS_GRAD, None, "dq_raw")
    G.compare(G.bf16_to_np(out["dk"]), P.l2norm_bwd(k, dk_), G.TOL_RMS_GRAD, None, "dk_raw")
    G.compare(da.cpu().numpy(), da_r, 1e-5, 1e-5, "da")
    G.compare(db.cpu().numpy(), db_r, 1e-5, 1e-5, "db")
    G.compare(ddt.cpu().numpy(), ddt_r, 1e-5, None, "ddt_bias")
    if mode == 1:
        G.compare(dA.cpu().numpy(), dA_r, 1e-5, None, "dA_log")


def test_prologue_end_to_end_through_the_operator():
    """Raw inputs -> prologue -> chunked forward and backward -> prologue
    backward, against the oracle chain (fp64 prologue, operands rounded to
    bf16 as on the device, fp64 recurrence and its reverse mode)."""
    import torch
    B, T, H, dk, dv = 2, 200, 2, 128, 64
    rows = B * T
    q, k, a, b, A_log, dtb = _inputs(rows, H, dk, seed=91)
    rng = np.random.default_rng(92)
    v = _f32(rng.standard_normal((B, T, H, dv)))
    d_out = _f32(rng.standard_normal((B, T, H, dv)))
    qo, ko, go, bo = _run_fwd(torch, q, k, a, b, A_log, dtb, 1, -5.0, 2.0)
    scale = dk ** -0.5
    shp = lambda x, d: x.view(B, T, H, d)  # noqa: E731
    vd, dod = _dev_bf16(v, torch), _dev_bf16(d_out, torch)
    out, _ = gdn.chunk_gated_delta_rule_fwd(shp(qo, dk), shp(ko, dk), vd, go.view(B, T, H),
                                            bo.view(B, T, H), scale=scale)
    r = gdn.chunk_gated_delta_rule_bwd(shp(qo, dk), shp(ko, dk), vd, go.view(B, T, H), bo.view(B, T, H),
                                       dod, scale=scale)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa: E731
    dq_raw = torch.empty((rows, H, dk), dtype=torch.bfloat16, device="cuda")
    dk_raw = torch.empty_like(dq_raw)
    da = torch.empty((rows, H), dtype=torch.float32, device="cuda")
    db = torch.empty_like(da)
    dA = torch.empty((H,), dtype=torch.float32, device="cuda")
    ddt = torch.empty_like(dA)
    gdn.gdn_prologue_bwd(_dev_bf16(q, torch), _dev_bf16(k, torch), t(a), t(b), t(A_log), t(dtb), 1,
                         -5.0, 2.0, r["dq"].view(rows, H, dk), r["dk"].view(rows, H, dk),
                         r["dg"].view(rows, H), r["dbeta"].view(rows, H), dq_raw, dk_raw, da, db, dA,
                         ddt, rows, H, dk)
    torch.cuda.synchronize()
    # oracle chain
    qh = _f32(P.l2norm(q)).reshape(B, T, H, dk)
    kh = _f32(P.l2norm(k)).reshape(B, T, H, dk)
    g_r, b_r = P.gates(a, b, A_log, dtb, mode="decay", beta_scale=2.0)
    wl = W.Workload(name="prologue", q=W.f32_to_bf16_bits(qh), k=W.f32_to_bf16_bits(kh),
                    v=W.f32_to_bf16_bits(v), g=g_r.astype(np.float32).reshape(B, T, H),
                    beta=W.f32_to_bf16_bits(b_r.reshape(B, T, H)), scale=scale,
                    d_out=W.f32_to_bf16_bits(d_out), d_final_state=np.zeros((B, H, dk, dv), np.float32))
    o_ref, _ = recurrence.workload_fwd(wl)
    G.compare(G.bf16_to_np(out), o_ref, G.TOL_RMS_IID, G.TOL_MAX_IID, "out")
    ref = recurrence.workload_bwd(wl)
    dq_r = P.l2norm_bwd(q, ref["dq"].reshape(rows, H, dk))
    dk_r = P.l2norm_bwd(k, ref["dk"].reshape(rows, H, dk))
    da_r, db_r, dA_r, ddt_r = P.gates_bwd(a, b, ref["dg"].reshape(rows, H), ref["dbeta"].reshape(rows, H),
                                          A_log, dtb, mode="decay", beta_scale=2.0)
    G.compare(G.bf16_to_np(dq_raw), dq_r, G.TOL_RMS_GRAD, None, "dq_raw")
    G.compare(G.bf16_to_np(dk_raw), dk_r, G.TOL_RMS_GRAD, None, "dk_raw")
    G.compare(da.cpu().numpy(), da_r, G.TOL_RMS_GRAD, None, "da")
    G.compare(db.cpu().numpy(), db_r, G.TOL_RMS_GRAD, None, "db")
    G.compare(ddt.cpu().numpy(), ddt_r, G.TOL_RMS_GRAD, None, "ddt_bias")
    G.compare(dA.cpu().numpy(), dA_r, G.TOL_RMS_GRAD, None, "dA_log")
    assert metrics.rel_l2(G.bf16_to_np(out), o_ref) < G.TOL_RMS_IID


@pytest.mark.parametrize("rows", [1, 5, 9])
def test_prologue_backward_head_sums_with_few_rows(rows):
    """The per-head sums split a head's rows over a cluster of CTAs; with fewer
    rows than parts some CTAs sum nothing and the totals must still be right."""
    import torch
    H, dk = 3, 64
    q, k, a, b, A_log, dtb = _inputs(max(rows, 4), H, dk, seed=60 + rows)
    q, k, a, b = q[:rows], k[:rows], a[:rows], b[:rows]
    rng = np.random.default_rng(61)
    dq = _f32(rng.standard_normal((rows, H, dk)))
    dk_ = _f32(rng.standard_normal((rows, H, dk)))
    dg = rng.standard_normal((rows, H)).astype(np.float32)
    dbeta = _f32(rng.standard_normal((rows, H)))
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa: E731
    out = {n: torch.empty((rows, H, dk), dtype=torch.bfloat16, device="cuda") for n in ("dq", "dk")}
    da = torch.empty((rows, H), dtype=torch.float32, device="cuda")
    db = torch.empty_like(da)
    dA = torch.empty((H,), dtype=torch.float32, device="cuda")
    ddt = torch.empty_like(dA)
    gdn.gdn_prologue_bwd(_dev_bf16(q, torch), _dev_bf16(k, torch), t(a), t(b), t(A_log), t(dtb), 1, -5.0, 1.0,
                         _dev_bf16(dq, torch), _dev_bf16(dk_, torch), t(dg), _dev_bf16(dbeta, torch),
                         out["dq"], out["dk"], da, db, dA, ddt, rows, H, dk)
    torch.cuda.synchronize()
    _, _, dA_r, ddt_r = P.gates_bwd(a, b, dg, dbeta, A_log, dtb, mode="decay", lower=-5.0, beta_scale=1.0)
    G.compare(ddt.cpu().numpy(), ddt_r, 1e-5, None, "ddt_bias")
    G.compare(dA.cpu().numpy(), dA_r, 1e-5, None, "dA_log")
