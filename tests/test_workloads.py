"""Seeded input generator and the oracle's whole-workload driver (CPU only)."""

import numpy as np
import torch

from linear_attention_sequence_chunked_gb300 import workloads as W
from oracle import recurrence


def test_bf16_rounding_matches_torch():
    r = np.random.default_rng(0)
    x = np.concatenate([r.standard_normal(100000).astype(np.float32) * 10,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3e-39, -7.5e5],
                                 dtype=np.float32)])
    ours = W.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = W.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_recipes_shapes_and_ranges():
    for cfg, kw in [(1, {}), (2, dict(T=128)), (3, dict(seqlens=[70, 58])), (4, dict(T=200)),
                    (5, dict(T=64, B=2, H=2, with_grad=True))]:
        wl = W.make_workload(cfg, **kw)
        k = wl.f32("k")
        assert np.allclose(np.linalg.norm(k, axis=-1), 1.0, atol=2e-2)
        assert np.all(wl.g <= 0)
        beta = wl.f32("beta")
        assert np.all(beta >= 0) and np.all(beta <= (2.0 if cfg == 5 else 1.0))
        if cfg == 4:
            assert np.all(wl.g == np.float32(-1e-3))
        if cfg == 3:
            assert np.all(wl.g >= -5.0)
            assert list(wl.cu_seqlens) == [0, 70, 128]
            qn = np.linalg.norm(wl.f32("q"), axis=-1)
            assert np.allclose(qn, 1.0, atol=2e-2)
    # determinism
    a = W.make_workload(2, T=64, B=1, H=2)
    b = W.make_workload(2, T=64, B=1, H=2)
    assert np.array_equal(a.q, b.q) and np.array_equal(a.g, b.g)


def test_config3_correlation():
    wl = W.make_workload(3, seqlens=[256], H=2)
    # q and k share the correlated sources: their cosine is clearly positive
    cos = np.sum(wl.f32("q") * wl.f32("k"), axis=-1)
    assert 0.3 < float(np.mean(cos)) < 0.7


def test_varlen_packed_equals_separate():
    """Packed sequences reset the state at each boundary: the oracle's packed
    result equals separate per-sequence runs exactly."""
    wl = W.random_workload(B=1, T=0, H=3, d_k=8, d_v=6, seed=7, seqlens=[5, 64, 1, 70],
                           initial_state=True)
    o, S = recurrence.workload_fwd(wl, threads=4)
    for s, (b, t0, t1) in enumerate(wl.seq_bounds()):
        for h in range(wl.H):
            oo, SS = recurrence.fwd_head(wl.f32("q")[0, t0:t1, h], wl.f32("k")[0, t0:t1, h],
                                         wl.f32("v")[0, t0:t1, h], wl.g[0, t0:t1, h],
                                         wl.f32("beta")[0, t0:t1, h], wl.scale,
                                         wl.initial_state[s, h])
            assert np.array_equal(oo, o[0, t0:t1, h])
            assert np.array_equal(SS, S[s, h])
