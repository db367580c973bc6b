"""The peak probes: the tcgen05 bf16 GEMM against a PyTorch fp32 product of
the same bf16 operands, and the copy bit for bit."""

import pytest

from linear_attention_sequence_chunked_gb300 import gdn

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 320), (2560, 2560, 1024), (1664, 768, 192)])
def test_gemm_probe_matches_torch(M, N, K):
    import torch
    g = torch.Generator(device="cuda").manual_seed(M + N + K)
    A = torch.randn((M, K), device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn((N, K), device="cuda", generator=g).to(torch.bfloat16)
    C = torch.full((M, N), float("nan"), device="cuda", dtype=torch.bfloat16)
    gdn.gdn_probe_gemm_bf16(A, B, C, M, N, K)
    st = gdn.gdn_get_last_device_error()
    assert st == 0, gdn.gdn_status_string(st)
    ref = A.float() @ B.float().T
    c = C.float()
    assert torch.isfinite(c).all(), "tiles left unwritten"
    err = (c - ref).norm() / ref.norm()
    assert err < 3e-3, float(err)                       # bf16 output rounding
    assert ((c - ref).abs().max() / ref.abs().max()) < 1e-2
    # the rounding is that of the exact fp32 sums: equal to torch's own rounding almost everywhere
    assert (C == ref.to(torch.bfloat16)).float().mean() > 0.95


def test_copy_probe_is_exact():
    import torch
    n = 16 * 1000003
    src = torch.randint(0, 255, (n,), dtype=torch.uint8, device="cuda")
    dst = torch.zeros_like(src)
    gdn.gdn_probe_copy(src, dst, n)
    torch.cuda.synchronize()
    assert torch.equal(src, dst)
