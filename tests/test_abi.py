"""The C ABI library: it builds, loads, exports every function that
include/gdn.h declares, and rejects bad arguments on the host before any
CUDA call (so these tests need no GPU)."""

import ctypes

import pytest

from linear_attention_sequence_chunked_gb300 import build, gdn


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gdn.load()


def test_exports_every_declared_function(lib):
    names = gdn.header_functions()
    assert set(names) >= {"gdn_chunk_fwd", "gdn_chunk_bwd", "gdn_chunk_fwd_workspace_size",
                          "gdn_chunk_bwd_workspace_size", "gdn_get_last_device_error",
                          "gdn_status_string"}
    raw = ctypes.CDLL(gdn.library_path())
    for n in names:
        assert hasattr(raw, n), n


def test_status_strings(lib):
    for code in range(7):
        s = gdn.gdn_status_string(code)
        assert s.startswith(gdn.STATUS_NAMES[code])
    assert gdn.gdn_status_string(99) == "GDN_ERR_UNKNOWN"


FAKE = 0x10000  # never dereferenced: every case below fails validation first


def _fwd(**over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, scale=1.0, initial_state=None,
                cu_seqlens=None, out=FAKE, final_state=None, B=1, T=64, H=1, d_k=64, d_v=64)
    args.update(over)
    lib = gdn.load()
    return lib.gdn_chunk_fwd(args["q"], args["k"], args["v"], args["g"], args["beta"],
                             args["scale"], args["initial_state"], args["cu_seqlens"], args["out"],
                             args["final_state"], args["B"], args["T"], args["H"], args["d_k"],
                             args["d_v"], None, 0, None)


@pytest.mark.parametrize("over,code", [
    (dict(d_k=96), 2), (dict(d_k=256), 2), (dict(d_v=32), 2), (dict(d_v=192), 2),
    (dict(B=0), 1), (dict(H=0), 1), (dict(T=-1), 1),
    (dict(q=None), 1), (dict(out=None), 1), (dict(beta=None), 1),
    (dict(k=FAKE + 2), 3), (dict(out=FAKE + 8), 3), (dict(final_state=FAKE + 4), 3),
    (dict(cu_seqlens=FAKE + 2), 3),
    (dict(B=70000), 2),
])
def test_forward_host_validation(lib, over, code):
    assert _fwd(**over) == code


@pytest.mark.parametrize("over,code", [
    (dict(d_k=96), 2), (dict(d_v=32), 2), (dict(B=0), 1), (dict(q=None), 1),
    (dict(out=None), 1), (dict(k=FAKE + 2), 3), (dict(final_state=FAKE + 4), 3),
])
def test_recurrent_host_validation(lib, over, code):
    args = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, scale=1.0, initial_state=None,
                cu_seqlens=None, out=FAKE, final_state=None, B=1, T=64, H=1, d_k=64, d_v=64)
    args.update(over)
    st = gdn.load().gdn_recurrent_fwd(args["q"], args["k"], args["v"], args["g"], args["beta"],
                                       args["scale"], args["initial_state"], args["cu_seqlens"],
                                       args["out"], args["final_state"], args["B"], args["T"],
                                       args["H"], args["d_k"], args["d_v"], None)
    assert st == code


@pytest.mark.parametrize("over,code", [
    (dict(d_k=96), 2), (dict(d_v=32), 2), (dict(B=0), 1), (dict(T=-1), 1), (dict(q=None), 1),
    (dict(g=None), 1), (dict(out=None), 1), (dict(k=FAKE + 2), 3), (dict(g=FAKE + 4), 3),
    (dict(final_state=FAKE + 4), 3), (dict(cu_seqlens=FAKE + 2), 3), (dict(H=70000), 2),
])
def test_kda_chunk_host_validation(lib, over, code):
    args = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, scale=1.0, initial_state=None,
                cu_seqlens=None, out=FAKE, final_state=None, B=1, T=64, H=1, d_k=64, d_v=64)
    args.update(over)
    st = gdn.load().gdn_kda_chunk_fwd(args["q"], args["k"], args["v"], args["g"], args["beta"],
                                       args["scale"], args["initial_state"], args["cu_seqlens"],
                                       args["out"], args["final_state"], args["B"], args["T"],
                                       args["H"], args["d_k"], args["d_v"], None, 0, None)
    assert st == code


def test_kda_chunk_workspace(lib):
    """The per-channel-gate forward's optional workspace: at d_k = 128 the
    tensor-core walk's operand block of every chunk (129 KB per chunk and
    head), at d_k = 64 T and P in fp32 (32 KB); a misaligned one is refused."""
    assert gdn.gdn_kda_chunk_fwd_workspace_size(4, 4096, 16, 128, 128, 0) == 4 * 64 * 16 * 132096
    assert gdn.gdn_kda_chunk_fwd_workspace_size(3, 200, 2, 64, 64, 1) == (200 // 64 + 3) * 2 * 32768
    assert gdn.gdn_kda_chunk_fwd_workspace_size(1, 64, 1, 96, 64, 0) == 0
    st = gdn.load().gdn_kda_chunk_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, None, None, FAKE, None,
                                       1, 64, 1, 64, 64, FAKE + 16, 1 << 20, None)
    assert st == 3


def test_kda_backward_host_validation(lib):
    l = gdn.load()
    B, T, H, K, V = 1, 128, 1, 64, 64
    need = gdn.gdn_kda_chunk_bwd_workspace_size(B, T, H, K, V, 0)
    # T and P, the start states and the end-state gradients of every chunk
    assert need == 2 * (32768 + 2 * 4 * K * V)
    assert gdn.gdn_kda_chunk_bwd_workspace_size(B, T, H, 96, V, 0) == 0

    def call(ws, ws_bytes, d_k=64, dq=FAKE, g=FAKE):
        return l.gdn_kda_chunk_bwd(FAKE, FAKE, FAKE, g, FAKE, 1.0, None, None, FAKE, None,
                                   dq, FAKE, FAKE, FAKE, FAKE, None, B, T, H, d_k, V, ws, ws_bytes, None)
    assert call(None, 0) == 1                   # workspace missing
    assert call(FAKE, need - 1) == 1            # workspace too small
    assert call(FAKE + 16, need) == 3           # workspace not 256-byte aligned
    assert call(FAKE, need, d_k=32) == 2
    assert call(FAKE, need, dq=None) == 1
    assert call(FAKE, need, g=FAKE + 4) == 3


def test_backward_host_validation(lib):
    l = gdn.load()
    need = gdn.gdn_chunk_bwd_workspace_size(1, 128, 1, 64, 64, 0)
    assert need > 0

    def call(ws, ws_bytes, d_k=64, dq=FAKE):
        return l.gdn_chunk_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, None, None, FAKE, None,
                               dq, FAKE, FAKE, FAKE, FAKE, None, 1, 128, 1, d_k, 64,
                               ws, ws_bytes, None)
    assert call(None, 0) == 1                   # workspace missing
    assert call(FAKE, need - 1) == 1            # workspace too small
    assert call(FAKE + 16, need) == 3           # workspace not 256-byte aligned
    assert call(FAKE, need, d_k=32) == 2
    assert call(FAKE, need, dq=None) == 1


def test_workspace_sizes(lib):
    assert gdn.gdn_chunk_fwd_workspace_size(4, 4096, 16, 128, 128, 0) >= 0
    a = gdn.gdn_chunk_bwd_workspace_size(4, 4096, 16, 128, 128, 0)
    b = gdn.gdn_chunk_bwd_workspace_size(4, 8192, 16, 128, 128, 0)
    assert b > a > 4 * 64 * 16 * 128 * 128 * 4  # at least one fp32 state per chunk
    assert gdn.gdn_chunk_bwd_workspace_size(1, 4096, 16, 96, 128, 0) == 0  # unsupported


def test_saved_route_sizes(lib):
    """The saved buffer is every chunk's fp32-sized start state then the T
    tiles; the saved-route workspace is the end-state gradients alone."""
    B, T, H, K, V = 4, 4096, 16, 128, 128
    chunks = B * T // 64
    state = 4 * K * V * chunks * H
    tiles = 16384 * chunks * H
    assert gdn.gdn_chunk_saved_size(B, T, H, K, V, 0) == state + tiles == 320 * 2**20
    assert gdn.gdn_chunk_bwd_saved_workspace_size(B, T, H, K, V, 0) == state
    # together they hold what the recomputing backward's workspace holds
    assert (gdn.gdn_chunk_saved_size(B, T, H, K, V, 0) + gdn.gdn_chunk_bwd_saved_workspace_size(B, T, H, K, V, 0)
            == gdn.gdn_chunk_bwd_workspace_size(B, T, H, K, V, 0))
    # packed: floor(T / 64) + N chunk slots
    assert gdn.gdn_chunk_bwd_saved_workspace_size(3, 200, 2, 64, 64, 1) == 256 * ((200 // 64 + 3) * 2 * 64 * 64 * 4 // 256)
    assert gdn.gdn_chunk_saved_size(1, 0, 1, 64, 64, 0) == 0
    assert gdn.gdn_chunk_saved_size(1, 64, 1, 96, 64, 0) == 0  # unsupported


def test_saved_route_host_validation(lib):
    l = gdn.load()
    need = gdn.gdn_chunk_saved_size(1, 128, 1, 64, 64, 0)
    wneed = gdn.gdn_chunk_bwd_saved_workspace_size(1, 128, 1, 64, 64, 0)
    assert need > 0 and wneed > 0

    def fwd(saved, nbytes, out=FAKE, d_k=64):
        return l.gdn_chunk_fwd_save(FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, None, None, out, None,
                                    1, 128, 1, d_k, 64, saved, nbytes, None)

    def bwd(saved, nbytes, ws=FAKE, ws_bytes=wneed, dq=FAKE, d_v=64):
        return l.gdn_chunk_bwd_saved(FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, None, FAKE, None,
                                     dq, FAKE, FAKE, FAKE, FAKE, None, 1, 128, 1, 64, d_v,
                                     saved, nbytes, ws, ws_bytes, None)
    assert fwd(None, 0) == 1                  # saved buffer missing
    assert fwd(FAKE, need - 1) == 1           # too small
    assert fwd(FAKE + 16, need) == 3          # not 256-byte aligned
    assert fwd(FAKE, need, out=None) == 1
    assert fwd(FAKE, need, d_k=32) == 2
    assert bwd(None, 0) == 1
    assert bwd(FAKE, need - 1) == 1
    assert bwd(FAKE + 64, need) == 3
    assert bwd(FAKE, need, ws=None, ws_bytes=0) == 1   # gradient workspace missing
    assert bwd(FAKE, need, ws_bytes=wneed - 1) == 1
    assert bwd(FAKE, need, ws=FAKE + 32) == 3
    assert bwd(FAKE, need, dq=None) == 1
    assert bwd(FAKE, need, d_v=48) == 2


def test_probe_host_validation(lib):
    l = gdn.load()
    assert l.gdn_probe_copy(FAKE, FAKE + 4096, 0, None) == 0          # nothing to do
    assert l.gdn_probe_copy(FAKE, FAKE + 4096, 24, None) == 1         # not a multiple of 16
    assert l.gdn_probe_copy(None, FAKE, 32, None) == 1
    assert l.gdn_probe_copy(FAKE + 8, FAKE + 4096, 32, None) == 3
    g = l.gdn_probe_gemm_bf16
    assert g(FAKE, FAKE, FAKE, 0, 256, 64, None) == 1
    assert g(FAKE, FAKE, FAKE, 192, 256, 64, None) == 2                 # M % 128
    assert g(FAKE, FAKE, FAKE, 128, 128, 64, None) == 2                 # N % 256
    assert g(FAKE, FAKE, FAKE, 128, 256, 96, None) == 2                 # K % 64
    assert g(FAKE, FAKE, FAKE, 128, 256, 65536 + 64, None) == 2
    assert g(None, FAKE, FAKE, 128, 256, 64, None) == 1
    assert g(FAKE, FAKE + 2, FAKE, 128, 256, 64, None) == 3


def test_split_host_validation(lib):
    l = gdn.load()
    need = gdn.gdn_chunk_fwd_split_workspace_size(2, 256, 2, 64, 64, 3)
    assert need > 0
    assert gdn.gdn_chunk_fwd_split_workspace_size(2, 256, 2, 64, 64, 0) == 0
    # more segments than chunks are clamped: the same layout as one segment per chunk
    assert (gdn.gdn_chunk_fwd_split_workspace_size(2, 256, 2, 64, 64, 99)
            == gdn.gdn_chunk_fwd_split_workspace_size(2, 256, 2, 64, 64, 4))

    def call(nseg=3, ws=FAKE, nbytes=need, out=FAKE, d_k=64):
        return l.gdn_chunk_fwd_split(FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, None, out, None, 2, 256, 2, d_k, 64,
                                     nseg, ws, nbytes, None)
    assert call(nseg=0) == 1
    assert call(ws=None, nbytes=0) == 1
    assert call(nbytes=need - 1) == 1
    assert call(ws=FAKE + 32) == 3
    assert call(out=None) == 1
    assert call(d_k=96) == 2


def test_tensor_arguments_must_be_dense_device_memory(lib):
    """The binding refuses a strided view or a host tensor before calling the
    library (the kernels would read either as dense device memory)."""
    import torch
    x = torch.zeros((1, 64, 1, 64), dtype=torch.bfloat16)
    g = torch.zeros((1, 64, 1, 64))
    beta = torch.zeros((1, 64, 1), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="contiguous"):
        gdn.gdn_kda_chunk_fwd(x.transpose(1, 3), x, x, g, beta, 1.0, None, None, x, None, 1, 64, 1, 64, 64)
    with pytest.raises(ValueError, match="CUDA"):
        gdn.gdn_kda_chunk_fwd(x, x, x, g, beta, 1.0, None, None, x, None, 1, 64, 1, 64, 64)
    with pytest.raises(ValueError, match="CUDA"):
        gdn.chunk_gated_delta_rule_fwd(x, x, x, g[..., 0], beta)


def test_wait_limit_entry_host_validation(lib):
    import ctypes
    f = lib.gdn_chunk_fwd_wait_limit
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_float] + [ctypes.c_void_p] * 4 + [ctypes.c_int] * 5 + \
        [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint32, ctypes.c_int, ctypes.c_void_p]
    f.restype = ctypes.c_int
    p = 1 << 20  # never dereferenced: every case is refused on the host
    # d_k = 64 is refused (its kernels keep the default bound), as is a missing workspace
    assert f(p, p, p, p, p, 1.0, None, None, p, None, 1, 128, 1, 64, 64, p, 1 << 20, 1, 0, None) == 2
    assert f(p, p, p, p, p, 1.0, None, None, p, None, 1, 128, 1, 128, 64, None, 0, 1, 0, None) == 2
    assert f(p, p, p, p, p, 1.0, None, None, p, None, 0, 128, 1, 128, 64, p, 1 << 20, 1, 0, None) == 1
