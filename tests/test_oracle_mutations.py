"""Plausible mistakes planted in a copy of the C oracle must each break a pin.

Every mutant is a textual edit of oracle/gdn_oracle.c (a dropped term, a
wrong sign, a wrong operand) compiled into a temporary library on the CPU.
The real oracle is never modified.
"""

import os

import pytest

from oracle import recurrence
from tests import pins

SRC = os.path.join(os.path.dirname(recurrence.__file__), "gdn_oracle.c")

# (name, original text, replacement, which occurrence to replace (0-based))
MUTANTS = [
    ("decay_dropped", "/* forget */\n        for (int i = 0; i < K * V; ++i) S[i] *= alpha;",
     "/* forget */\n        for (int i = 0; i < K * V; ++i) S[i] *= 1.0;", 0),
    ("error_sign", "(vt[j] - v_old[j])", "(vt[j] + v_old[j])", 0),
    ("beta_dropped", "S[(size_t)i * V + j] += b * kt[i] * (vt[j] - v_old[j]);",
     "S[(size_t)i * V + j] += kt[i] * (vt[j] - v_old[j]);", 0),
    ("read_with_query", "acc += S[(size_t)i * V + j] * kt[i];\n            v_old[j] = acc;",
     "acc += S[(size_t)i * V + j] * qt[i];\n            v_old[j] = acc;", 0),
    ("scale_dropped", "o[(size_t)t * V + j] = scale * acc;", "o[(size_t)t * V + j] = acc;", 0),
    ("matrix_form_write_beta_dropped", "Rn[(size_t)r * K + c] = acc + b * vt[r] * kt[c];",
     "Rn[(size_t)r * K + c] = acc + vt[r] * kt[c];", 0),
    ("bwd_dk_sign", "dk[(size_t)t * K + i] = b * a1 - a2;", "dk[(size_t)t * K + i] = b * a1 + a2;", 0),
    ("bwd_dg_dropped", "dg[t] = acc;", "dg[t] = 0.0;", 0),
    ("bwd_de_beta_dropped", "de[j] = b * acc;", "de[j] = acc;", 0),
    ("bwd_decay_dropped", "dS[(size_t)i * V + j] = alpha * d;", "dS[(size_t)i * V + j] = d;", 0),
    ("bwd_dbeta_sign", "dbeta[t] = acc;", "dbeta[t] = -acc;", 0),
    ("bwd_dq_scale", "dq[(size_t)t * K + i] = scale * acc;", "dq[(size_t)t * K + i] = acc;", 0),
    ("bwd_dS_operand", "dS[(size_t)i * V + j] += scale * qt[i] * dot[j];",
     "dS[(size_t)i * V + j] += scale * kt[i] * dot[j];", 0),
    ("bwd_dv_wrong", "dv[(size_t)t * V + j] = de[j];", "dv[(size_t)t * V + j] = e[j];", 0),
]


def _apply(text, old, new, occ):
    idx = -1
    for _ in range(occ + 1):
        idx = text.index(old, idx + 1)
    return text[:idx] + new + text[idx + len(old):]


@pytest.mark.parametrize("name,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, occ):
    with open(SRC) as f:
        text = f.read()
    mutated = _apply(text, old, new, occ)
    assert mutated != text
    src = tmp_path / f"{name}.c"
    src.write_text(mutated)
    lib = recurrence.OracleLib(recurrence.build_oracle(force=True, src=str(src),
                                                       out=str(tmp_path / f"{name}.so")))
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
