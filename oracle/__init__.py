"""CPU oracle for the gated delta rule -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import, call, link or execute anything in this package.  The
CUDA operator never does, and shares no code with it.

* ``recurrence`` -- fp64 per-token recurrence (C, via ctypes): forward in the
  page-1 loop form and the page-4 matrix form, plus a hand-derived reverse mode.
* ``chunked``    -- fp64 chunked WY algebra (numpy): forward and reverse mode.
* ``metrics``    -- error metrics (relative RMS / L2, max-relative, windows).
"""
