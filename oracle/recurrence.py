"""Python front end of the fp64 recurrence oracle -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package's smoke check and the benchmark's CPU-baseline
leg may import this module.  It loads ``gdn_oracle.c`` (compiled with plain
gcc, no architecture flags) through ctypes and runs it once per
(sequence, head) on fp64 copies of the bf16-rounded inputs.  ctypes releases
the GIL during each call, so a thread pool spreads (sequence, head) units over
the host cores.

Definitions followed: "Research Sprint Day 1", section "The GDN update" (the
per-token loop) and "Research Sprint Day 2 - Rooflines", GDN update equation
(the matrix form); see ``gdn_oracle.c`` for the exact statements.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


def build_oracle(force: bool = False, src: str = _SRC, out: str = _SO) -> str:
    """Compile the C oracle (``src``) into a shared library (``out``)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c99",
                           "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def _ptr(a):
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(_dp)


def _c64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


class OracleLib:
    """One loaded copy of the C oracle.  All arrays are fp64; one
    (sequence, head) per call."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i, d = ctypes.c_int, ctypes.c_double
        lib.gdn_oracle_fwd.argtypes = [i, i, i, d] + [_dp] * 8
        lib.gdn_oracle_fwd.restype = i
        lib.gdn_oracle_fwd_matrix_form.argtypes = [i, i, i, d] + [_dp] * 8
        lib.gdn_oracle_fwd_matrix_form.restype = i
        lib.gdn_oracle_bwd.argtypes = [i, i, i, d] + [_dp] * 14
        lib.gdn_oracle_bwd.restype = i
        self._lib = lib
        self.path = path

    def fwd_head(self, q, k, v, g, beta, scale, S0=None):
        """Page-1 loop.  q, k (T,K); v (T,V); g, beta (T,); S0 (K,V) or None.
        Returns (o (T,V), S_final (K,V))."""
        q, k, v, g, beta, S0 = map(_c64, (q, k, v, g, beta, S0))
        T, K = q.shape
        V = v.shape[1]
        o = np.zeros((T, V))
        S = np.zeros((K, V))
        rc = self._lib.gdn_oracle_fwd(T, K, V, float(scale), _ptr(q), _ptr(k), _ptr(v),
                                      _ptr(g), _ptr(beta), _ptr(S0), _ptr(o), _ptr(S))
        if rc != 0:
            raise MemoryError("oracle allocation failed")
        return o, S

    def fwd_head_matrix_form(self, q, k, v, g, beta, scale, R0=None):
        """Page-4 matrix form; state R is (V,K).  Returns (o (T,V), R_final (V,K))."""
        q, k, v, g, beta, R0 = map(_c64, (q, k, v, g, beta, R0))
        T, K = q.shape
        V = v.shape[1]
        o = np.zeros((T, V))
        R = np.zeros((V, K))
        rc = self._lib.gdn_oracle_fwd_matrix_form(T, K, V, float(scale), _ptr(q), _ptr(k),
                                                  _ptr(v), _ptr(g), _ptr(beta), _ptr(R0),
                                                  _ptr(o), _ptr(R))
        if rc != 0:
            raise MemoryError("oracle allocation failed")
        return o, R

    def bwd_head(self, q, k, v, g, beta, scale, S0, dO, dS_final):
        """Reverse mode of the page-1 loop.  Returns dict of dq, dk, dv, dg,
        dbeta, dS0."""
        q, k, v, g, beta, S0, dO, dS_final = map(
            _c64, (q, k, v, g, beta, S0, dO, dS_final))
        T, K = q.shape
        V = v.shape[1]
        out = dict(dq=np.zeros((T, K)), dk=np.zeros((T, K)), dv=np.zeros((T, V)),
                   dg=np.zeros(T), dbeta=np.zeros(T), dS0=np.zeros((K, V)))
        rc = self._lib.gdn_oracle_bwd(T, K, V, float(scale), _ptr(q), _ptr(k), _ptr(v),
                                      _ptr(g), _ptr(beta), _ptr(S0), _ptr(dO),
                                      _ptr(dS_final), _ptr(out["dq"]), _ptr(out["dk"]),
                                      _ptr(out["dv"]), _ptr(out["dg"]), _ptr(out["dbeta"]),
                                      _ptr(out["dS0"]))
        if rc != 0:
            raise MemoryError("oracle allocation failed")
        return out


def _load() -> OracleLib:
    global _lib
    with _lock:
        if _lib is None:
            _lib = OracleLib(build_oracle())
    return _lib


def fwd_head(*args, **kw):
    return _load().fwd_head(*args, **kw)


def fwd_head_matrix_form(*args, **kw):
    return _load().fwd_head_matrix_form(*args, **kw)


def bwd_head(*args, **kw):
    return _load().bwd_head(*args, **kw)


# ----------------------------------------------------------------------------
# whole-workload entry points
# ----------------------------------------------------------------------------

def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _units(wl, units):
    if units is None:
        return [(s, h) for s in range(wl.n_seq) for h in range(wl.H)]
    return list(units)


def workload_fwd(wl, units=None, threads=None):
    """Run the oracle forward on (sequence, head) ``units`` of a Workload.

    Returns (o, S): o is fp64 with v's shape (rows of units not computed are
    NaN); S is fp64 (n_seq, H, K, V) (NaN where not computed).
    """
    units = _units(wl, units)
    q32, k32, v32, beta32 = wl.f32("q"), wl.f32("k"), wl.f32("v"), wl.f32("beta")
    g32 = wl.g
    o = np.full(wl.v.shape, np.nan)
    S = np.full((wl.n_seq, wl.H, wl.d_k, wl.d_v), np.nan)
    bounds = wl.seq_bounds()

    def run(unit):
        s, h = unit
        b, t0, t1 = bounds[s]
        S0 = None if wl.initial_state is None else wl.initial_state[s, h]
        oo, SS = fwd_head(q32[b, t0:t1, h], k32[b, t0:t1, h], v32[b, t0:t1, h],
                          g32[b, t0:t1, h], beta32[b, t0:t1, h], wl.scale, S0)
        o[b, t0:t1, h] = oo
        S[s, h] = SS

    with ThreadPoolExecutor(max_workers=threads or default_threads()) as ex:
        list(ex.map(run, units))
    return o, S


def workload_bwd(wl, units=None, threads=None):
    """Oracle gradients on ``units``.  Returns dict of fp64 arrays shaped like
    the inputs (dq, dk, dv (B,T,H,d); dg, dbeta (B,T,H); dS0 (N,H,K,V));
    entries of units not computed are NaN."""
    units = _units(wl, units)
    q32, k32, v32, beta32 = wl.f32("q"), wl.f32("k"), wl.f32("v"), wl.f32("beta")
    dO32 = wl.f32("d_out")
    g32 = wl.g
    res = dict(dq=np.full(wl.q.shape, np.nan), dk=np.full(wl.k.shape, np.nan),
               dv=np.full(wl.v.shape, np.nan), dg=np.full(wl.g.shape, np.nan),
               dbeta=np.full(wl.g.shape, np.nan),
               dS0=np.full((wl.n_seq, wl.H, wl.d_k, wl.d_v), np.nan))
    bounds = wl.seq_bounds()

    def run(unit):
        s, h = unit
        b, t0, t1 = bounds[s]
        S0 = None if wl.initial_state is None else wl.initial_state[s, h]
        dSf = None if wl.d_final_state is None else wl.d_final_state[s, h]
        r = bwd_head(q32[b, t0:t1, h], k32[b, t0:t1, h], v32[b, t0:t1, h],
                     g32[b, t0:t1, h], beta32[b, t0:t1, h], wl.scale, S0,
                     dO32[b, t0:t1, h], dSf)
        res["dq"][b, t0:t1, h] = r["dq"]
        res["dk"][b, t0:t1, h] = r["dk"]
        res["dv"][b, t0:t1, h] = r["dv"]
        res["dg"][b, t0:t1, h] = r["dg"]
        res["dbeta"][b, t0:t1, h] = r["dbeta"]
        res["dS0"][s, h] = r["dS0"]

    with ThreadPoolExecutor(max_workers=threads or default_threads()) as ex:
        list(ex.map(run, units))
    return res
