"""fp64 prologue of the gated delta rule: q/k L2 normalisation and the two
gates, with their reverse mode -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg use this
module; the CUDA library shares no code with it.

Forward, per (token, head), following "Research Sprint Day 2 - Rooflines",
GDN layer pseudocode steps 4 and 5:
  q_hat = q / sqrt(|q|^2 + eps),  k_hat likewise        (step 4, per row)
  beta  = c * sigmoid(b),  c = 1, or 2 with negative eigenvalues allowed
  g     = -exp(A_log[h]) * softplus(a + dt_bias[h])      (decay gate, <= 0)
or, for the bounded gates that fla issue #1550 runs its CP2 test with
(lower bound -5),
  g     = lower * sigmoid(a + dt_bias[h])                (in (lower, 0))
Readings (the pages are silent): eps = 1e-6 inside the square root, so that
an all-zero row maps to zero instead of NaN; dt_bias defaults to 0 in the
bounded form.

Reverse mode (hand-derived; pinned by finite differences in tests):
  with r = (|x|^2 + eps)^-1/2 and y = r x:   dx = r (dy - y (y . dy))
  db = dbeta * c * s (1 - s),  s = sigmoid(b)
  decay:   da = dg * (-exp(A_log) * sigmoid(u)),  u = a + dt_bias
           dA_log[h] = sum over (b, t) of dg * g,  ddt_bias[h] = sum of da
  bounded: da = dg * lower * s_u (1 - s_u),  s_u = sigmoid(u);  ddt_bias[h] = sum of da
"""

from __future__ import annotations

import numpy as np

EPS = 1e-6


def sigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    return np.where(x >= 0, 1.0 / (1.0 + np.exp(-np.abs(x))), np.exp(-np.abs(x)) / (1.0 + np.exp(-np.abs(x))))


def softplus(x):
    x = np.asarray(x, dtype=np.float64)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def l2norm(x):
    """Rows of the last axis scaled to unit length (with EPS)."""
    x = np.asarray(x, dtype=np.float64)
    r = 1.0 / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + EPS)
    return x * r


def l2norm_bwd(x, dy):
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    r = 1.0 / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + EPS)
    y = x * r
    return r * (dy - y * np.sum(y * dy, axis=-1, keepdims=True))


def gates(a, b, A_log=None, dt_bias=None, mode="decay", lower=-5.0, beta_scale=1.0):
    """(g, beta) from the raw gate inputs a, b of shape (..., H); A_log and
    dt_bias have shape (H,)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    H = a.shape[-1]
    dtb = np.zeros(H) if dt_bias is None else np.asarray(dt_bias, dtype=np.float64)
    u = a + dtb
    if mode == "decay":
        g = -np.exp(np.asarray(A_log, dtype=np.float64)) * softplus(u)
    elif mode == "bounded":
        g = lower * sigmoid(u)
    else:
        raise ValueError(mode)
    beta = beta_scale * sigmoid(b)
    return g, beta


def gates_bwd(a, b, dg, dbeta, A_log=None, dt_bias=None, mode="decay", lower=-5.0, beta_scale=1.0):
    """(da, db, dA_log, ddt_bias); the per-head sums run over every axis but the last."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    dg = np.asarray(dg, dtype=np.float64)
    dbeta = np.asarray(dbeta, dtype=np.float64)
    H = a.shape[-1]
    dtb = np.zeros(H) if dt_bias is None else np.asarray(dt_bias, dtype=np.float64)
    u = a + dtb
    axes = tuple(range(a.ndim - 1))
    sb = sigmoid(b)
    db = dbeta * beta_scale * sb * (1.0 - sb)
    su = sigmoid(u)
    if mode == "decay":
        e = np.exp(np.asarray(A_log, dtype=np.float64))
        g = -e * softplus(u)
        da = dg * (-e * su)
        dA_log = np.sum(dg * g, axis=axes)
    else:
        da = dg * lower * su * (1.0 - su)
        dA_log = None
    ddt_bias = np.sum(da, axis=axes)
    return da, db, dA_log, ddt_bias
