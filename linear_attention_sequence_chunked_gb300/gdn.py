"""Thin Python binding of the C ABI in include/gdn.h.

Every function here only marshals arguments (tensor -> device pointer,
stream -> handle) and checks the returned status; all arithmetic runs in the
CUDA kernels of ``_build/libgdn.so``.  There is no CPU fallback: if the
library is missing or no GPU is present, calls raise.

Low-level names mirror the C ABI (gdn_chunk_fwd, gdn_chunk_bwd, ...).  The
two convenience wrappers (chunk_gated_delta_rule_fwd / _bwd) allocate the
outputs and the workspace with torch and then call the same entry points.
"""

from __future__ import annotations

import ctypes
import os
import re
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

GDN_OK = 0
STATUS_NAMES = {
    0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED", 3: "GDN_ERR_MISALIGNED",
    4: "GDN_ERR_BAD_SEQLENS", 5: "GDN_ERR_TIMEOUT", 6: "GDN_ERR_CUDA",
}
HEADER = os.path.join(_build.ROOT, "include", "gdn.h")


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


def library_path() -> str:
    return _build.LIB


def header_functions():
    """Names of the functions declared in include/gdn.h."""
    with open(HEADER) as f:
        text = f.read()
    return re.findall(r"GDN_API\s+[\w\s\*]+?\b(gdn_\w+)\s*\(", text)


def load():
    """Load the built library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built: {path} is missing (run build())")
        lib = ctypes.CDLL(path)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.gdn_status_string.argtypes = [i]
        lib.gdn_status_string.restype = ctypes.c_char_p
        lib.gdn_chunk_fwd_workspace_size.argtypes = [i] * 6
        lib.gdn_chunk_fwd_workspace_size.restype = sz
        lib.gdn_chunk_bwd_workspace_size.argtypes = [i] * 6
        lib.gdn_chunk_bwd_workspace_size.restype = sz
        lib.gdn_chunk_fwd.argtypes = [vp] * 5 + [f] + [vp] * 4 + [i] * 5 + [vp, sz, vp]
        lib.gdn_chunk_fwd.restype = i
        lib.gdn_chunk_bwd.argtypes = [vp] * 5 + [f] + [vp] * 10 + [i] * 5 + [vp, sz, vp]
        lib.gdn_chunk_bwd.restype = i
        lib.gdn_recurrent_fwd.argtypes = [vp] * 5 + [f] + [vp] * 4 + [i] * 5 + [vp]
        lib.gdn_recurrent_fwd.restype = i
        lib.gdn_kda_recurrent_fwd.argtypes = [vp] * 5 + [f] + [vp] * 4 + [i] * 5 + [vp]
        lib.gdn_kda_recurrent_fwd.restype = i
        lib.gdn_kda_chunk_fwd_workspace_size.argtypes = [i] * 6
        lib.gdn_kda_chunk_fwd_workspace_size.restype = sz
        lib.gdn_kda_chunk_fwd.argtypes = [vp] * 5 + [f] + [vp] * 4 + [i] * 5 + [vp, sz, vp]
        lib.gdn_kda_chunk_fwd.restype = i
        lib.gdn_kda_chunk_bwd_workspace_size.argtypes = [i] * 6
        lib.gdn_kda_chunk_bwd_workspace_size.restype = sz
        lib.gdn_kda_chunk_bwd.argtypes = [vp] * 5 + [f] + [vp] * 10 + [i] * 5 + [vp, sz, vp]
        lib.gdn_kda_chunk_bwd.restype = i
        lib.gdn_prologue_fwd.argtypes = [vp] * 6 + [i, f, f] + [vp] * 4 + [i] * 3 + [vp]
        lib.gdn_prologue_fwd.restype = i
        lib.gdn_prologue_bwd.argtypes = [vp] * 6 + [i, f, f] + [vp] * 10 + [i] * 3 + [vp]
        lib.gdn_prologue_bwd.restype = i
        lib.gdn_get_last_device_error.argtypes = [vp]
        lib.gdn_get_last_device_error.restype = i
        lib.gdn_chunk_saved_size.argtypes = [i] * 6
        lib.gdn_chunk_saved_size.restype = sz
        lib.gdn_chunk_bwd_saved_workspace_size.argtypes = [i] * 6
        lib.gdn_chunk_bwd_saved_workspace_size.restype = sz
        lib.gdn_chunk_fwd_save.argtypes = [vp] * 5 + [f] + [vp] * 4 + [i] * 5 + [vp, sz, vp]
        lib.gdn_chunk_fwd_save.restype = i
        lib.gdn_chunk_bwd_saved.argtypes = [vp] * 5 + [f] + [vp] * 9 + [i] * 5 + [vp, sz, vp, sz, vp]
        lib.gdn_chunk_bwd_saved.restype = i
        lib.gdn_chunk_bwd_saved_wait_limit.argtypes = ([vp] * 5 + [f] + [vp] * 9 + [i] * 5
                                                       + [vp, sz, vp, sz, ctypes.c_uint32, i, vp])
        lib.gdn_chunk_bwd_saved_wait_limit.restype = i
        lib.gdn_chunk_fwd_split_workspace_size.argtypes = [i] * 6
        lib.gdn_chunk_fwd_split_workspace_size.restype = sz
        lib.gdn_chunk_fwd_split.argtypes = [vp] * 5 + [f] + [vp] * 3 + [i] * 6 + [vp, sz, vp]
        lib.gdn_chunk_fwd_split.restype = i
        lib.gdn_probe_copy.argtypes = [vp, vp, sz, vp]
        lib.gdn_probe_copy.restype = i
        lib.gdn_probe_gemm_bf16.argtypes = [vp, vp, vp, i, i, i, vp]
        lib.gdn_probe_gemm_bf16.restype = i
        lib.gdn_chunk_bwd_noalloc.argtypes = [vp] * 5 + [f] + [vp] * 10 + [i] * 5 + [vp]
        lib.gdn_chunk_bwd_noalloc.restype = i
        lib.gdn_chunk_fwd_wait_limit.argtypes = [vp] * 5 + [f] + [vp] * 4 + [i] * 5 + [vp, sz, ctypes.c_uint32, i, vp]
        lib.gdn_chunk_fwd_wait_limit.restype = i
        lib.gdn_kernel_launches.argtypes = []
        lib.gdn_kernel_launches.restype = ctypes.c_uint64
        _lib = lib
        return lib


def _ptr(x):
    """Device address of a tensor argument (None and raw integer addresses
    pass through).  The kernels read every tensor as dense row-major device
    memory, so a strided view or a host tensor is refused here, before any
    call into the library."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_contiguous():
        raise ValueError(f"expected a contiguous tensor, got shape {tuple(x.shape)} strides {x.stride()}")
    if x.device.type != "cuda":
        raise ValueError(f"expected a CUDA tensor, got one on {x.device}")
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, where: str):
    if status != GDN_OK:
        raise GdnError(status, where)


# ----------------------------------------------------------------------------
# C ABI mirrors
# ----------------------------------------------------------------------------

def gdn_status_string(status: int) -> str:
    return load().gdn_status_string(int(status)).decode()


def gdn_chunk_fwd_workspace_size(B, T, H, d_k, d_v, varlen) -> int:
    return int(load().gdn_chunk_fwd_workspace_size(B, T, H, d_k, d_v, int(bool(varlen))))


def gdn_chunk_bwd_workspace_size(B, T, H, d_k, d_v, varlen) -> int:
    return int(load().gdn_chunk_bwd_workspace_size(B, T, H, d_k, d_v, int(bool(varlen))))


def gdn_chunk_fwd(q, k, v, g, beta, scale, initial_state, cu_seqlens, out, final_state,
                  B, T, H, d_k, d_v, workspace=None, workspace_bytes=0, stream=None):
    st = load().gdn_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                              _ptr(initial_state), _ptr(cu_seqlens), _ptr(out),
                              _ptr(final_state), B, T, H, d_k, d_v, _ptr(workspace),
                              int(workspace_bytes), _stream(stream))
    _check(st, "gdn_chunk_fwd")


def gdn_chunk_fwd_wait_limit(q, k, v, g, beta, scale, initial_state, cu_seqlens, out, final_state,
                             B, T, H, d_k, d_v, workspace, workspace_bytes, wait_limit, stall_first_wait=0,
                             stream=None):
    """gdn_chunk_fwd with a chosen bound (polls) on the kernels' hand-off
    waits, and optionally a first wait that nothing ends: for exercising
    failure detection."""
    st = load().gdn_chunk_fwd_wait_limit(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                         _ptr(initial_state), _ptr(cu_seqlens), _ptr(out),
                                         _ptr(final_state), B, T, H, d_k, d_v, _ptr(workspace),
                                         int(workspace_bytes), int(wait_limit), int(stall_first_wait),
                                         _stream(stream))
    _check(st, "gdn_chunk_fwd_wait_limit")


def gdn_chunk_bwd(q, k, v, g, beta, scale, initial_state, cu_seqlens, d_out, d_final_state,
                  dq, dk, dv, dg, dbeta, d_initial_state, B, T, H, d_k, d_v,
                  workspace=None, workspace_bytes=0, stream=None):
    st = load().gdn_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                              _ptr(initial_state), _ptr(cu_seqlens), _ptr(d_out),
                              _ptr(d_final_state), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg),
                              _ptr(dbeta), _ptr(d_initial_state), B, T, H, d_k, d_v,
                              _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check(st, "gdn_chunk_bwd")


def gdn_chunk_saved_size(B, T, H, d_k, d_v, varlen) -> int:
    return int(load().gdn_chunk_saved_size(B, T, H, d_k, d_v, int(bool(varlen))))


def gdn_chunk_bwd_saved_workspace_size(B, T, H, d_k, d_v, varlen) -> int:
    return int(load().gdn_chunk_bwd_saved_workspace_size(B, T, H, d_k, d_v, int(bool(varlen))))


def gdn_chunk_fwd_save(q, k, v, g, beta, scale, initial_state, cu_seqlens, out, final_state,
                       B, T, H, d_k, d_v, saved, saved_bytes, stream=None):
    st = load().gdn_chunk_fwd_save(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                   _ptr(initial_state), _ptr(cu_seqlens), _ptr(out),
                                   _ptr(final_state), B, T, H, d_k, d_v, _ptr(saved),
                                   int(saved_bytes), _stream(stream))
    _check(st, "gdn_chunk_fwd_save")


def gdn_chunk_bwd_saved(q, k, v, g, beta, scale, cu_seqlens, d_out, d_final_state,
                        dq, dk, dv, dg, dbeta, d_initial_state, B, T, H, d_k, d_v,
                        saved, saved_bytes, workspace=None, workspace_bytes=0, stream=None):
    st = load().gdn_chunk_bwd_saved(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                    _ptr(cu_seqlens), _ptr(d_out), _ptr(d_final_state), _ptr(dq),
                                    _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta),
                                    _ptr(d_initial_state), B, T, H, d_k, d_v, _ptr(saved),
                                    int(saved_bytes), _ptr(workspace), int(workspace_bytes),
                                    _stream(stream))
    _check(st, "gdn_chunk_bwd_saved")


def gdn_chunk_bwd_saved_wait_limit(q, k, v, g, beta, scale, cu_seqlens, d_out, d_final_state,
                                   dq, dk, dv, dg, dbeta, d_initial_state, B, T, H, d_k, d_v,
                                   saved, saved_bytes, workspace, workspace_bytes, wait_limit,
                                   stall_first_wait=0, stream=None):
    """gdn_chunk_bwd_saved with a chosen bound (polls) on the gradient pass's
    hand-off waits, and optionally a first wait that nothing ends: for
    exercising failure detection."""
    st = load().gdn_chunk_bwd_saved_wait_limit(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                               _ptr(cu_seqlens), _ptr(d_out), _ptr(d_final_state), _ptr(dq),
                                               _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta),
                                               _ptr(d_initial_state), B, T, H, d_k, d_v, _ptr(saved),
                                               int(saved_bytes), _ptr(workspace), int(workspace_bytes),
                                               int(wait_limit), int(stall_first_wait), _stream(stream))
    _check(st, "gdn_chunk_bwd_saved_wait_limit")


def gdn_chunk_fwd_split_workspace_size(B, T, H, d_k, d_v, nseg) -> int:
    return int(load().gdn_chunk_fwd_split_workspace_size(B, T, H, d_k, d_v, nseg))


def gdn_chunk_fwd_split(q, k, v, g, beta, scale, initial_state, out, final_state, B, T, H, d_k, d_v, nseg,
                        workspace, workspace_bytes, stream=None):
    st = load().gdn_chunk_fwd_split(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                    _ptr(initial_state), _ptr(out), _ptr(final_state), B, T, H, d_k, d_v,
                                    int(nseg), _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check(st, "gdn_chunk_fwd_split")


def gdn_probe_copy(src, dst, nbytes, stream=None):
    _check(load().gdn_probe_copy(_ptr(src), _ptr(dst), int(nbytes), _stream(stream)), "gdn_probe_copy")


def gdn_probe_gemm_bf16(A, B, C, M, N, K, stream=None):
    _check(load().gdn_probe_gemm_bf16(_ptr(A), _ptr(B), _ptr(C), M, N, K, _stream(stream)),
           "gdn_probe_gemm_bf16")


def gdn_recurrent_fwd(q, k, v, g, beta, scale, initial_state, cu_seqlens, out, final_state,
                      B, T, H, d_k, d_v, stream=None):
    st = load().gdn_recurrent_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                  _ptr(initial_state), _ptr(cu_seqlens), _ptr(out),
                                  _ptr(final_state), B, T, H, d_k, d_v, _stream(stream))
    _check(st, "gdn_recurrent_fwd")


def gdn_kda_recurrent_fwd(q, k, v, g, beta, scale, initial_state, cu_seqlens, out, final_state,
                          B, T, H, d_k, d_v, stream=None):
    st = load().gdn_kda_recurrent_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                      _ptr(initial_state), _ptr(cu_seqlens), _ptr(out),
                                      _ptr(final_state), B, T, H, d_k, d_v, _stream(stream))
    _check(st, "gdn_kda_recurrent_fwd")


def gdn_kda_chunk_fwd_workspace_size(B, T, H, d_k, d_v, varlen) -> int:
    return int(load().gdn_kda_chunk_fwd_workspace_size(B, T, H, d_k, d_v, int(bool(varlen))))


def gdn_kda_chunk_bwd_workspace_size(B, T, H, d_k, d_v, varlen) -> int:
    return int(load().gdn_kda_chunk_bwd_workspace_size(B, T, H, d_k, d_v, int(bool(varlen))))


def gdn_kda_chunk_fwd(q, k, v, g, beta, scale, initial_state, cu_seqlens, out, final_state,
                      B, T, H, d_k, d_v, workspace=None, workspace_bytes=0, stream=None):
    st = load().gdn_kda_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                  _ptr(initial_state), _ptr(cu_seqlens), _ptr(out),
                                  _ptr(final_state), B, T, H, d_k, d_v, _ptr(workspace),
                                  int(workspace_bytes), _stream(stream))
    _check(st, "gdn_kda_chunk_fwd")


def gdn_kda_chunk_bwd(q, k, v, g, beta, scale, initial_state, cu_seqlens, d_out, d_final_state,
                      dq, dk, dv, dg, dbeta, d_initial_state, B, T, H, d_k, d_v,
                      workspace=None, workspace_bytes=0, stream=None):
    st = load().gdn_kda_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                  _ptr(initial_state), _ptr(cu_seqlens), _ptr(d_out),
                                  _ptr(d_final_state), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg),
                                  _ptr(dbeta), _ptr(d_initial_state), B, T, H, d_k, d_v,
                                  _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check(st, "gdn_kda_chunk_bwd")


def chunk_kda_fwd(q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None, stream=None):
    """Allocate out, the final state and the per-chunk workspace and run
    gdn_kda_chunk_fwd: q, k (B, T, H, d_k) bf16; v (B, T, H, d_v) bf16;
    g (B, T, H, d_k) fp32 (one log decay per key channel); beta (B, T, H)
    bf16.  Returns (out, final_state)."""
    import torch
    _validate(q, k, v, g, beta, initial_state, cu_seqlens, per_channel_gate=True)
    B, T, H, d_k, d_v = _dims(q, v, cu_seqlens)
    if scale is None:
        scale = d_k ** -0.5
    out = torch.empty(v.shape, dtype=torch.bfloat16, device=v.device)
    fs = torch.empty((B, H, d_k, d_v), dtype=torch.float32, device=v.device)
    nbytes = gdn_kda_chunk_fwd_workspace_size(B, T, H, d_k, d_v, cu_seqlens is not None)
    ws = _workspace(nbytes, v.device)
    gdn_kda_chunk_fwd(q, k, v, g, beta, scale, initial_state, cu_seqlens, out, fs, B, T, H, d_k, d_v,
                      ws, nbytes, stream)
    return out, fs


def chunk_kda_bwd(q, k, v, g, beta, d_out, scale=None, initial_state=None, cu_seqlens=None,
                  d_final_state=None, stream=None):
    """Allocate gradients and the workspace and run gdn_kda_chunk_bwd (the
    per-channel-gate backward).  Returns a dict of dq, dk, dv, dg (per key
    channel, fp32), dbeta and d_initial_state."""
    import torch
    _validate(q, k, v, g, beta, initial_state, cu_seqlens, d_out=d_out, d_final_state=d_final_state,
              per_channel_gate=True)
    B, T, H, d_k, d_v = _dims(q, v, cu_seqlens)
    if scale is None:
        scale = d_k ** -0.5
    dev = v.device
    res = dict(dq=torch.empty(q.shape, dtype=torch.bfloat16, device=dev),
               dk=torch.empty(k.shape, dtype=torch.bfloat16, device=dev),
               dv=torch.empty(v.shape, dtype=torch.bfloat16, device=dev),
               dg=torch.empty(g.shape, dtype=torch.float32, device=dev),
               dbeta=torch.empty(beta.shape, dtype=torch.bfloat16, device=dev),
               d_initial_state=torch.empty((B, H, d_k, d_v), dtype=torch.float32, device=dev))
    nbytes = gdn_kda_chunk_bwd_workspace_size(B, T, H, d_k, d_v, cu_seqlens is not None)
    ws = _workspace(nbytes, dev)
    gdn_kda_chunk_bwd(q, k, v, g, beta, scale, initial_state, cu_seqlens, d_out, d_final_state,
                      res["dq"], res["dk"], res["dv"], res["dg"], res["dbeta"], res["d_initial_state"],
                      B, T, H, d_k, d_v, ws, nbytes, stream)
    return res


def gdn_prologue_fwd(q_raw, k_raw, a, b, A_log, dt_bias, gate_mode, lower, beta_scale,
                     q, k, g, beta, rows, H, d_k, stream=None):
    st = load().gdn_prologue_fwd(_ptr(q_raw), _ptr(k_raw), _ptr(a), _ptr(b), _ptr(A_log),
                                 _ptr(dt_bias), int(gate_mode), float(lower), float(beta_scale),
                                 _ptr(q), _ptr(k), _ptr(g), _ptr(beta), rows, H, d_k, _stream(stream))
    _check(st, "gdn_prologue_fwd")


def gdn_prologue_bwd(q_raw, k_raw, a, b, A_log, dt_bias, gate_mode, lower, beta_scale,
                     dq, dk, dg, dbeta, dq_raw, dk_raw, da, db, dA_log, ddt_bias, rows, H, d_k,
                     stream=None):
    st = load().gdn_prologue_bwd(_ptr(q_raw), _ptr(k_raw), _ptr(a), _ptr(b), _ptr(A_log),
                                 _ptr(dt_bias), int(gate_mode), float(lower), float(beta_scale),
                                 _ptr(dq), _ptr(dk), _ptr(dg), _ptr(dbeta), _ptr(dq_raw),
                                 _ptr(dk_raw), _ptr(da), _ptr(db), _ptr(dA_log), _ptr(ddt_bias),
                                 rows, H, d_k, _stream(stream))
    _check(st, "gdn_prologue_bwd")


def gdn_chunk_bwd_noalloc(q, k, v, g, beta, scale, initial_state, cu_seqlens, d_out, d_final_state,
                          dq, dk, dv, dg, dbeta, d_initial_state, B, T, H, d_k, d_v, stream=None):
    """gdn_chunk_bwd without a workspace argument: for callers that may not
    allocate device memory, the scratch comes from a fixed array inside the
    library (GDN_NOALLOC_SCRATCH_BYTES).  Calls that overlap on the GPU race."""
    st = load().gdn_chunk_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                      _ptr(initial_state), _ptr(cu_seqlens), _ptr(d_out),
                                      _ptr(d_final_state), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg),
                                      _ptr(dbeta), _ptr(d_initial_state), B, T, H, d_k, d_v,
                                      _stream(stream))
    _check(st, "gdn_chunk_bwd_noalloc")


def gdn_get_last_device_error(stream=None) -> int:
    return int(load().gdn_get_last_device_error(_stream(stream)))


def gdn_kernel_launches() -> int:
    return int(load().gdn_kernel_launches())


# ----------------------------------------------------------------------------
# convenience wrappers (torch tensors in, torch tensors out)
# ----------------------------------------------------------------------------

def _dims(q, v, cu_seqlens):
    Bq, T, H, d_k = q.shape
    d_v = v.shape[-1]
    if cu_seqlens is not None:
        if Bq != 1:
            raise ValueError("packed inputs must have batch extent 1")
        B = int(cu_seqlens.numel()) - 1
    else:
        B = Bq
    return B, T, H, d_k, d_v


def _validate(q, k, v, g, beta, initial_state=None, cu_seqlens=None, d_out=None,
              d_final_state=None, per_channel_gate=False):
    """Dtype, shape and device checks of the convenience wrappers, before any
    library call: the kernels read each tensor with a fixed element type and
    extent, so a mismatch would otherwise read past a buffer or give silent
    garbage."""
    import torch
    if q.dim() != 4:
        raise ValueError(f"q must be (B, T, H, d_k), got shape {tuple(q.shape)}")
    Bq, T, H, d_k = q.shape
    want = [("q", q, torch.bfloat16, (Bq, T, H, d_k)),
            ("k", k, torch.bfloat16, (Bq, T, H, d_k)),
            ("v", v, torch.bfloat16, None),
            ("g", g, torch.float32, (Bq, T, H, d_k) if per_channel_gate else (Bq, T, H)),
            ("beta", beta, torch.bfloat16, (Bq, T, H))]
    if v.dim() != 4 or tuple(v.shape[:3]) != (Bq, T, H):
        raise ValueError(f"v must be (B, T, H, d_v) with q's (B, T, H), got {tuple(v.shape)}")
    d_v = v.shape[3]
    if cu_seqlens is not None:
        if cu_seqlens.dtype != torch.int32:
            raise ValueError(f"cu_seqlens must be int32, got {cu_seqlens.dtype}")
        if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
            raise ValueError("cu_seqlens must be a 1-D tensor of N + 1 offsets")
        N = cu_seqlens.numel() - 1
        want.append(("cu_seqlens", cu_seqlens, torch.int32, (N + 1,)))
    else:
        N = Bq
    if initial_state is not None:
        want.append(("initial_state", initial_state, torch.float32, (N, H, d_k, d_v)))
    if d_out is not None:
        want.append(("d_out", d_out, torch.bfloat16, (Bq, T, H, d_v)))
    if d_final_state is not None:
        want.append(("d_final_state", d_final_state, torch.float32, (N, H, d_k, d_v)))
    for name, t, dtype, shape in want:
        if t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
        if shape is not None and tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
        if t.device != q.device:
            raise ValueError(f"{name} is on {t.device}, q on {q.device}: all tensors must share one device")


def _workspace(nbytes, device):
    import torch
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def chunk_gated_delta_rule_fwd(q, k, v, g, beta, scale=None, initial_state=None,
                               cu_seqlens=None, output_final_state=True, stream=None,
                               save_for_backward=False):
    """Allocate outputs and run gdn_chunk_fwd.  Returns (out, final_state), or
    (out, final_state, saved) with save_for_backward: gdn_chunk_fwd_save, whose
    `saved` buffer chunk_gated_delta_rule_bwd(..., saved=saved) reuses."""
    import torch
    _validate(q, k, v, g, beta, initial_state, cu_seqlens)
    B, T, H, d_k, d_v = _dims(q, v, cu_seqlens)
    if scale is None:
        scale = d_k ** -0.5
    out = torch.empty(v.shape, dtype=torch.bfloat16, device=v.device)
    fs = (torch.empty((B, H, d_k, d_v), dtype=torch.float32, device=v.device)
          if output_final_state else None)
    if save_for_backward:
        nbytes = gdn_chunk_saved_size(B, T, H, d_k, d_v, cu_seqlens is not None)
        saved = torch.empty(nbytes, dtype=torch.uint8, device=v.device)
        gdn_chunk_fwd_save(q, k, v, g, beta, scale, initial_state, cu_seqlens, out, fs,
                           B, T, H, d_k, d_v, saved, nbytes, stream)
        return out, fs, saved
    nbytes = gdn_chunk_fwd_workspace_size(B, T, H, d_k, d_v, cu_seqlens is not None)
    ws = _workspace(nbytes, v.device)
    gdn_chunk_fwd(q, k, v, g, beta, scale, initial_state, cu_seqlens, out, fs,
                  B, T, H, d_k, d_v, ws, nbytes, stream)
    return out, fs


def chunk_gated_delta_rule_fwd_split(q, k, v, g, beta, nseg, scale=None, initial_state=None,
                                     output_final_state=True, stream=None):
    """Allocate outputs and run gdn_chunk_fwd_split (dense inputs, every
    sequence as nseg segments).  Returns (out, final_state)."""
    import torch
    _validate(q, k, v, g, beta, initial_state)
    B, T, H, d_k, d_v = _dims(q, v, None)
    if scale is None:
        scale = d_k ** -0.5
    out = torch.empty(v.shape, dtype=torch.bfloat16, device=v.device)
    fs = (torch.empty((B, H, d_k, d_v), dtype=torch.float32, device=v.device)
          if output_final_state else None)
    nbytes = gdn_chunk_fwd_split_workspace_size(B, T, H, d_k, d_v, nseg)
    ws = _workspace(nbytes, v.device)
    gdn_chunk_fwd_split(q, k, v, g, beta, scale, initial_state, out, fs, B, T, H, d_k, d_v, nseg,
                        ws, nbytes, stream)
    return out, fs


def chunk_gated_delta_rule_bwd(q, k, v, g, beta, d_out, scale=None, initial_state=None,
                               cu_seqlens=None, d_final_state=None, stream=None, saved=None):
    """Allocate gradients and run gdn_chunk_bwd, or gdn_chunk_bwd_saved when
    `saved` (from chunk_gated_delta_rule_fwd(..., save_for_backward=True) on
    the same inputs) is given.  Returns a dict of tensors."""
    import torch
    _validate(q, k, v, g, beta, initial_state, cu_seqlens, d_out=d_out, d_final_state=d_final_state)
    if saved is not None and (saved.dtype != torch.uint8 or saved.device != q.device):
        raise ValueError("saved must be the uint8 buffer that the saving forward returned, on q's device")
    B, T, H, d_k, d_v = _dims(q, v, cu_seqlens)
    if scale is None:
        scale = d_k ** -0.5
    dev = v.device
    res = dict(dq=torch.empty(q.shape, dtype=torch.bfloat16, device=dev),
               dk=torch.empty(k.shape, dtype=torch.bfloat16, device=dev),
               dv=torch.empty(v.shape, dtype=torch.bfloat16, device=dev),
               dg=torch.empty(g.shape, dtype=torch.float32, device=dev),
               dbeta=torch.empty(beta.shape, dtype=torch.bfloat16, device=dev),
               d_initial_state=torch.empty((B, H, d_k, d_v), dtype=torch.float32, device=dev))
    if saved is not None:
        nbytes = gdn_chunk_bwd_saved_workspace_size(B, T, H, d_k, d_v, cu_seqlens is not None)
        ws = _workspace(nbytes, dev)
        gdn_chunk_bwd_saved(q, k, v, g, beta, scale, cu_seqlens, d_out, d_final_state,
                            res["dq"], res["dk"], res["dv"], res["dg"], res["dbeta"],
                            res["d_initial_state"], B, T, H, d_k, d_v, saved, saved.numel(),
                            ws, nbytes, stream)
        return res
    nbytes = gdn_chunk_bwd_workspace_size(B, T, H, d_k, d_v, cu_seqlens is not None)
    ws = _workspace(nbytes, dev)
    gdn_chunk_bwd(q, k, v, g, beta, scale, initial_state, cu_seqlens, d_out, d_final_state,
                  res["dq"], res["dk"], res["dv"], res["dg"], res["dbeta"],
                  res["d_initial_state"], B, T, H, d_k, d_v, ws, nbytes, stream)
    return res


# ----------------------------------------------------------------------------
# autograd: the training route behind torch.autograd
# ----------------------------------------------------------------------------

def _autograd_function():
    import torch

    class _ChunkGatedDeltaRule(torch.autograd.Function):
        """Forward: gdn_chunk_fwd_save (the output, the final state, and every
        chunk's start state and T tiles kept for the backward).  Backward:
        gdn_chunk_bwd_saved from them."""

        @staticmethod
        def forward(ctx, q, k, v, g, beta, initial_state, scale, cu_seqlens):
            out, fs, saved = chunk_gated_delta_rule_fwd(q, k, v, g, beta, scale=scale,
                                                        initial_state=initial_state,
                                                        cu_seqlens=cu_seqlens, save_for_backward=True)
            ctx.save_for_backward(q, k, v, g, beta, saved)
            ctx.scale = scale
            ctx.cu_seqlens = cu_seqlens
            ctx.has_initial_state = initial_state is not None
            return out, fs

        @staticmethod
        def backward(ctx, d_out, d_fs):
            q, k, v, g, beta, saved = ctx.saved_tensors
            if d_out is None:
                d_out = torch.zeros_like(v)
            d_out = d_out.to(torch.bfloat16).contiguous()
            d_fs = None if d_fs is None else d_fs.to(torch.float32).contiguous()
            r = chunk_gated_delta_rule_bwd(q, k, v, g, beta, d_out, scale=ctx.scale,
                                           cu_seqlens=ctx.cu_seqlens, d_final_state=d_fs, saved=saved)
            d_s0 = r["d_initial_state"] if ctx.has_initial_state else None
            return r["dq"], r["dk"], r["dv"], r["dg"], r["dbeta"], d_s0, None, None

    return _ChunkGatedDeltaRule


_AUTOGRAD = None


def chunk_gated_delta_rule(q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None):
    """The chunked gated delta rule with autograd: (B, T, H, d_k) bf16 q, k;
    (B, T, H, d_v) bf16 v; (B, T, H) fp32 g and bf16 beta; optional fp32
    initial state (N, H, d_k, d_v) and int32 cu_seqlens (packed inputs, B = 1).
    Returns (out (B, T, H, d_v) bf16, final_state (N, H, d_k, d_v) fp32); the
    backward runs from the chunk states the forward kept (gradients w.r.t.
    q, k, v, g, beta and initial_state, in their dtypes)."""
    global _AUTOGRAD
    if _AUTOGRAD is None:
        _AUTOGRAD = _autograd_function()
    _validate(q, k, v, g, beta, initial_state, cu_seqlens)
    if scale is None:
        scale = q.shape[-1] ** -0.5
    return _AUTOGRAD.apply(q, k, v, g, beta, initial_state, float(scale), cu_seqlens)
