"""Error metrics used to compare a result with the oracle -- TEST INFRASTRUCTURE.

* rel_l2 (== relative RMS): ||x - r||_2 / max(||r||_2, 1e-30), the metric of
  the cuLA issue #126 reproduction (rel_l2 with a 1e-30 clamp) and the
  "Relative RMS output error" of fla issue #1550.
* max_rel: max|x - r| / max|r| over the whole tensor.  The "max relative error
  across all elements" of "Research Sprint Day 1" is undefined elementwise
  near r = 0; this per-tensor normalisation is the reading used here.
* window_rel_l2: rel_l2 per token window (8 windows, the last one taking the
  remainder), as in the cuLA reproduction's per-window report.
"""

import numpy as np


def rel_l2(x, r):
    x = np.asarray(x, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    return float(np.linalg.norm((x - r).ravel()) / max(np.linalg.norm(r.ravel()), 1e-30))


def max_rel(x, r):
    x = np.asarray(x, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    return float(np.max(np.abs(x - r)) / max(np.max(np.abs(r)), 1e-30))


def window_rel_l2(x, r, axis=1, windows=8):
    x = np.asarray(x, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    T = x.shape[axis]
    w = T // windows
    out = []
    for i in range(windows):
        lo = i * w
        hi = T if i == windows - 1 else (i + 1) * w
        sl = [slice(None)] * x.ndim
        sl[axis] = slice(lo, hi)
        out.append(rel_l2(x[tuple(sl)], r[tuple(sl)]))
    return out
