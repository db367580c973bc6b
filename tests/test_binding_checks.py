"""The convenience wrappers check dtypes, shapes and devices before any
library call (CPU only: the checks need no GPU and no library)."""

import pytest

torch = pytest.importorskip("torch")

from linear_attention_sequence_chunked_gb300 import gdn  # noqa: E402


def _good(B=2, T=8, H=3, dk=64, dv=128, varlen=False):
    bf, f32 = torch.bfloat16, torch.float32
    Bq = 1 if varlen else B
    t = dict(q=torch.zeros(Bq, T, H, dk, dtype=bf), k=torch.zeros(Bq, T, H, dk, dtype=bf),
             v=torch.zeros(Bq, T, H, dv, dtype=bf), g=torch.zeros(Bq, T, H, dtype=f32),
             beta=torch.zeros(Bq, T, H, dtype=bf),
             initial_state=torch.zeros(B, H, dk, dv, dtype=f32),
             cu_seqlens=torch.tensor([0, 3, T], dtype=torch.int32) if varlen else None,
             d_out=torch.zeros(Bq, T, H, dv, dtype=bf),
             d_final_state=torch.zeros(B, H, dk, dv, dtype=f32))
    return t


def _call(t, **kw):
    gdn._validate(t["q"], t["k"], t["v"], t["g"], t["beta"], t["initial_state"], t["cu_seqlens"],
                  d_out=t["d_out"], d_final_state=t["d_final_state"], **kw)


@pytest.mark.parametrize("varlen", [False, True])
def test_valid_arguments_pass(varlen):
    _call(_good(varlen=varlen))


BAD = [
    ("q", lambda t: t["q"].float(), "q must be torch.bfloat16"),
    ("k", lambda t: t["k"].half(), "k must be torch.bfloat16"),
    ("g", lambda t: t["g"].bfloat16(), "g must be torch.float32"),
    ("beta", lambda t: t["beta"].float(), "beta must be torch.bfloat16"),
    ("initial_state", lambda t: t["initial_state"].bfloat16(), "initial_state must be torch.float32"),
    ("d_out", lambda t: t["d_out"].float(), "d_out must be torch.bfloat16"),
    ("d_final_state", lambda t: t["d_final_state"].double(), "d_final_state must be torch.float32"),
    ("k", lambda t: t["k"][:, :, :2].contiguous(), "k must have shape"),
    ("v", lambda t: t["v"][:, :4].contiguous(), "v must be (B, T, H, d_v)"),
    ("g", lambda t: t["g"][..., None].contiguous(), "g must have shape"),
    ("beta", lambda t: t["beta"][:, :5].contiguous(), "beta must have shape"),
    ("initial_state", lambda t: t["initial_state"][:, :, :32].contiguous(), "initial_state must have shape"),
    ("d_out", lambda t: t["d_out"][..., :64].contiguous(), "d_out must have shape"),
]


@pytest.mark.parametrize("name,edit,msg", BAD, ids=[f"{b[0]}-{i}" for i, b in enumerate(BAD)])
def test_mismatch_raises_before_any_library_call(name, edit, msg):
    t = _good()
    t[name] = edit(t)
    with pytest.raises(ValueError, match=msg.replace("(", r"\(").replace(")", r"\)")):
        _call(t)


def test_cu_seqlens_must_be_int32():
    t = _good(varlen=True)
    t["cu_seqlens"] = t["cu_seqlens"].long()
    with pytest.raises(ValueError, match="cu_seqlens must be int32"):
        _call(t)


def test_packed_state_count_follows_cu_seqlens():
    t = _good(varlen=True)
    t["initial_state"] = torch.zeros(1, 3, 64, 128)  # 2 sequences in cu_seqlens
    with pytest.raises(ValueError, match="initial_state must have shape"):
        _call(t)


def test_per_channel_gate_shape():
    t = _good()
    with pytest.raises(ValueError, match="g must have shape"):
        _call(t, per_channel_gate=True)
    t["g"] = torch.zeros(2, 8, 3, 64)
    _call(t, per_channel_gate=True)


def test_wrappers_validate_first():
    t = _good()
    t["g"] = t["g"].bfloat16()
    with pytest.raises(ValueError, match="g must be torch.float32"):
        gdn.chunk_gated_delta_rule_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"])
    with pytest.raises(ValueError, match="g must be torch.float32"):
        gdn.chunk_gated_delta_rule_bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["d_out"])
    with pytest.raises(ValueError, match="g must be torch.float32"):
        gdn.chunk_gated_delta_rule(t["q"], t["k"], t["v"], t["g"], t["beta"])
