"""Seeded synthetic inputs for the chunked gated delta rule operator.

This module only draws random numbers and shapes them into the five workloads
used by the tests and the benchmark.  It contains none of the operator's own
arithmetic (no decay products, no recurrence, no chunk algebra), so that the
CUDA path and the CPU oracle can both consume it without sharing any of the
method's code.

Recipes (per workload, draw order q, k, v, gates, dO):

1. "single head": B=1, H=1, T=256, d_k=d_v=64.  q, v ~ N(0,1); k ~ N(0,1)
   then L2-normalised per row; beta = sigmoid(N(0,1)); g = logsigmoid(N(0,1)+2).
2. "dense sweep": B=4, H=16, T in {256,1024,4096}, (d_k,d_v) in
   {(64,64),(64,128),(128,128)}.  q, v ~ N(0,1); k L2-normalised;
   beta = sigmoid(N(0,1)); g = -exp(A_log) * softplus(a + dt_bias) with
   a ~ N(0,1) per (b,t,h), A_log ~ U(0, ln 16) per head, dt_bias ~ U(-1,1)
   per head.  (Research Sprint Day 2 -- Rooflines, GDN layer pseudocode,
   step 5 "the two gates".)
3. "correlated varlen": two packed sequences of 5120 tokens, H=12,
   d_k=d_v=128.  c, n1, n2, n3 ~ N(0,1); c' = 0.8 c + 0.6 n3 (correlation
   0.8); q = 0.7 c + 0.3 n1, k = 0.7 c' + 0.3 n2, both L2-normalised in fp32
   before the bf16 cast; g = -5 sigmoid(N(0,1)); beta = sigmoid(N(0,1));
   v ~ N(0,1).  (fla issue #1550, "Reproduction and evidence": asymmetric Q/K,
   bounded gates with lower bound -5, sequence lengths [5120, 5120].)
4. "slow decay": B=1, T=65536, H=16, d_k=d_v=128.  q, v ~ N(0,1); k
   L2-normalised; g = -1e-3 constant; beta = sigmoid(N(0,1) - 2).
   (cuLA issue #126: 64K slow-decay heads.)
5. "training": B=8, T=4096, H=16, d_k=128, d_v=256.  As 2 but
   beta = 2 sigmoid(N(0,1)) in (0,2) ("allow_neg_eigval"); dO ~ N(0,1).

All floating inputs are drawn in fp32; q, k, v, beta and dO are rounded to
bf16 with round-to-nearest-even, g stays fp32.  Both the oracle and the GPU
consume the rounded values.  Seeds: workload 1 uses seed 0 and workload n
(n >= 2) uses seed n, unless overridden.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np


# ----------------------------------------------------------------------------
# bf16 helpers (bit patterns stored as uint16)
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round-to-nearest-even); returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to fp32 exactly."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return (1.0 / (1.0 + np.exp(-x.astype(np.float64)))).astype(np.float32)


def _logsigmoid(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.float64)
    return (np.minimum(x, 0.0) - np.log1p(np.exp(-np.abs(x)))).astype(np.float32)


def _softplus(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.float64)
    return (np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))).astype(np.float32)


def _l2norm_rows(x: np.ndarray) -> np.ndarray:
    """L2-normalise the last axis in fp32 (the input preparation step)."""
    x = x.astype(np.float32)
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True, dtype=np.float32))
    return (x / np.maximum(n, np.float32(1e-12))).astype(np.float32)


# ----------------------------------------------------------------------------
# Workload container
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class Workload:
    """One batch of operator inputs.

    Dense layout: q, k (B,T,H,d_k); v (B,T,H,d_v); g, beta (B,T,H).
    Packed layout (cu_seqlens set): B == 1 in the arrays, N = len(cu_seqlens)-1
    sequences; states are (N,H,d_k,d_v).
    bf16 tensors are uint16 bit patterns; g and states are fp32.
    """

    name: str
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    g: np.ndarray
    beta: np.ndarray
    scale: float
    initial_state: Optional[np.ndarray] = None
    cu_seqlens: Optional[np.ndarray] = None
    d_out: Optional[np.ndarray] = None
    d_final_state: Optional[np.ndarray] = None

    @property
    def B(self) -> int:
        return int(self.q.shape[0])

    @property
    def T(self) -> int:
        return int(self.q.shape[1])

    @property
    def H(self) -> int:
        return int(self.q.shape[2])

    @property
    def d_k(self) -> int:
        return int(self.q.shape[3])

    @property
    def d_v(self) -> int:
        return int(self.v.shape[3])

    @property
    def n_seq(self) -> int:
        if self.cu_seqlens is not None:
            return int(len(self.cu_seqlens) - 1)
        return self.B

    def seq_bounds(self):
        """List of (batch_index, t_begin, t_end) for every sequence."""
        if self.cu_seqlens is None:
            return [(b, 0, self.T) for b in range(self.B)]
        cu = [int(x) for x in self.cu_seqlens]
        return [(0, cu[i], cu[i + 1]) for i in range(len(cu) - 1)]

    @property
    def token_heads(self) -> int:
        return self.B * self.T * self.H

    # fp32 views of the bf16 inputs (exact)
    def f32(self, name: str) -> np.ndarray:
        arr = getattr(self, name)
        if arr is None:
            return None
        if arr.dtype == np.uint16:
            return bf16_bits_to_f32(arr).reshape(arr.shape)
        return arr.astype(np.float32)


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(seed))


def _normal(rng, shape):
    return rng.standard_normal(size=shape, dtype=np.float32)


def _dense_gates(rng, B, T, H):
    """g = -exp(A_log) * softplus(a + dt_bias), per (b,t,h)."""
    a = _normal(rng, (B, T, H))
    A_log = rng.uniform(0.0, math.log(16.0), size=(H,)).astype(np.float32)
    dt_bias = rng.uniform(-1.0, 1.0, size=(H,)).astype(np.float32)
    g = -np.exp(A_log.astype(np.float64))[None, None, :] * _softplus(a + dt_bias[None, None, :])
    return g.astype(np.float32)


def make_workload(config: int, *, T: Optional[int] = None, B: Optional[int] = None,
                  H: Optional[int] = None, d_k: Optional[int] = None,
                  d_v: Optional[int] = None, seqlens=None, seed: Optional[int] = None,
                  with_grad: bool = False, initial_state: bool = False) -> Workload:
    """Build workload ``config`` (1..5) with optional size overrides.

    Size overrides keep the value recipe of the workload and only change the
    shapes, so that small parity cases and the full-size cases share a recipe.
    ``seqlens`` (list of ints) turns the workload into a packed one.
    ``initial_state`` draws a non-zero fp32 initial state ~ N(0,1)/sqrt(d_k)
    after all other draws; ``with_grad`` draws dO ~ N(0,1) (bf16) last.
    """
    defaults = {
        1: dict(B=1, T=256, H=1, d_k=64, d_v=64),
        2: dict(B=4, T=4096, H=16, d_k=128, d_v=128),
        3: dict(B=1, T=10240, H=12, d_k=128, d_v=128),
        4: dict(B=1, T=65536, H=16, d_k=128, d_v=128),
        5: dict(B=8, T=4096, H=16, d_k=128, d_v=256),
    }[config]
    B = defaults["B"] if B is None else B
    T = defaults["T"] if T is None else T
    H = defaults["H"] if H is None else H
    d_k = defaults["d_k"] if d_k is None else d_k
    d_v = defaults["d_v"] if d_v is None else d_v
    if config == 3 and seqlens is None and T == defaults["T"]:
        seqlens = [5120, 5120]
    if seqlens is not None:
        seqlens = [int(s) for s in seqlens]
        T = int(sum(seqlens))
        B = 1
    if seed is None:
        seed = 0 if config == 1 else config
    rng = _rng(seed)

    shp_k = (B, T, H, d_k)
    shp_v = (B, T, H, d_v)
    if config == 3:
        c = _normal(rng, shp_k)
        n1 = _normal(rng, shp_k)
        n2 = _normal(rng, shp_k)
        n3 = _normal(rng, shp_k)
        cp = np.float32(0.8) * c + np.float32(0.6) * n3
        q = _l2norm_rows(np.float32(0.7) * c + np.float32(0.3) * n1)
        k = _l2norm_rows(np.float32(0.7) * cp + np.float32(0.3) * n2)
        v = _normal(rng, shp_v)
        g = (-5.0 * _sigmoid(_normal(rng, (B, T, H)))).astype(np.float32)
        beta = _sigmoid(_normal(rng, (B, T, H)))
    else:
        q = _normal(rng, shp_k)
        k = _l2norm_rows(_normal(rng, shp_k))
        v = _normal(rng, shp_v)
        if config == 1:
            beta = _sigmoid(_normal(rng, (B, T, H)))
            g = _logsigmoid(_normal(rng, (B, T, H)) + np.float32(2.0))
        elif config == 2:
            beta = _sigmoid(_normal(rng, (B, T, H)))
            g = _dense_gates(rng, B, T, H)
        elif config == 4:
            g = np.full((B, T, H), -1e-3, dtype=np.float32)
            beta = _sigmoid(_normal(rng, (B, T, H)) - np.float32(2.0))
        elif config == 5:
            beta = (2.0 * _sigmoid(_normal(rng, (B, T, H)))).astype(np.float32)
            g = _dense_gates(rng, B, T, H)
        else:
            raise ValueError(f"unknown workload {config}")

    n_seq = len(seqlens) if seqlens is not None else B
    s0 = None
    if initial_state:
        s0 = (_normal(rng, (n_seq, H, d_k, d_v)) / np.float32(math.sqrt(d_k))).astype(np.float32)
    d_out = None
    d_fs = None
    if with_grad:
        d_out = f32_to_bf16_bits(_normal(rng, shp_v)).reshape(shp_v)
        d_fs = np.zeros((n_seq, H, d_k, d_v), dtype=np.float32)

    cu = None
    if seqlens is not None:
        cu = np.zeros(len(seqlens) + 1, dtype=np.int32)
        cu[1:] = np.cumsum(seqlens)

    return Workload(
        name=f"config{config}",
        q=f32_to_bf16_bits(q).reshape(shp_k),
        k=f32_to_bf16_bits(k).reshape(shp_k),
        v=f32_to_bf16_bits(v).reshape(shp_v),
        g=np.ascontiguousarray(g, dtype=np.float32),
        beta=f32_to_bf16_bits(beta).reshape((B, T, H)),
        scale=float(d_k) ** -0.5,
        initial_state=s0,
        cu_seqlens=cu,
        d_out=d_out,
        d_final_state=d_fs,
    )


def random_workload(*, B, T, H, d_k, d_v, seed, seqlens=None, beta_max=1.0,
                    g_low=-0.5, initial_state=False, with_grad=False,
                    d_final_state=False) -> Workload:
    """Generic iid workload for edge-case tests (any shape, optional packing).

    q, v ~ N(0,1); k L2-normalised; beta = beta_max * U(0,1); g ~ U(g_low, 0).
    """
    rng = _rng(seed)
    if seqlens is not None:
        seqlens = [int(s) for s in seqlens]
        T = int(sum(seqlens))
        B = 1
    shp_k = (B, T, H, d_k)
    shp_v = (B, T, H, d_v)
    q = _normal(rng, shp_k)
    k = _l2norm_rows(_normal(rng, shp_k))
    v = _normal(rng, shp_v)
    beta = (beta_max * rng.uniform(0.0, 1.0, size=(B, T, H))).astype(np.float32)
    g = rng.uniform(g_low, 0.0, size=(B, T, H)).astype(np.float32)
    n_seq = len(seqlens) if seqlens is not None else B
    s0 = None
    if initial_state:
        s0 = (_normal(rng, (n_seq, H, d_k, d_v)) / np.float32(math.sqrt(d_k))).astype(np.float32)
    d_out = d_fs = None
    if with_grad:
        d_out = f32_to_bf16_bits(_normal(rng, shp_v)).reshape(shp_v)
        if d_final_state:
            d_fs = _normal(rng, (n_seq, H, d_k, d_v)).astype(np.float32)
        else:
            d_fs = np.zeros((n_seq, H, d_k, d_v), dtype=np.float32)
    cu = None
    if seqlens is not None:
        cu = np.zeros(len(seqlens) + 1, dtype=np.int32)
        cu[1:] = np.cumsum(seqlens)
    return Workload(
        name="random",
        q=f32_to_bf16_bits(q).reshape(shp_k),
        k=f32_to_bf16_bits(k).reshape(shp_k),
        v=f32_to_bf16_bits(v).reshape(shp_v),
        g=g,
        beta=f32_to_bf16_bits(beta).reshape((B, T, H)),
        scale=float(d_k) ** -0.5,
        initial_state=s0,
        cu_seqlens=cu,
        d_out=d_out,
        d_final_state=d_fs,
    )
