"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Each mutant is a textual edit of ``oracle/pda_oracle.c`` compiled into a
temporary library on the CPU; the real oracle source is never modified.  This
shows the pins would catch a dropped term, a wrong sign, a wrong index or a
transposed operand.  Every mutant keeps all memory accesses in bounds.
"""
import os

import pytest

import oracle
import oracle_pins

MUTANTS = {
    "interleaved head map": ("const int32_t kvh = h / G;", "const int32_t kvh = h % P->Hkv;"),
    "scale dropped": ("s[t] = P->scale * dot;", "s[t] = dot;"),
    "no max subtraction": ("s[t] = exp(s[t] - mx);", "s[t] = exp(s[t]);"),
    "exp sign flipped": ("s[t] = exp(s[t] - mx);", "s[t] = exp(mx - s[t]);"),
    "no normalisation": ("out[d] /= z;", "out[d] /= 1.0;"),
    "values used as keys": ("const uint16_t* krow = P->k_pool +", "const uint16_t* krow = P->v_pool +"),
    "keys used as values": ("const uint16_t* vrow = P->v_pool +", "const uint16_t* vrow = P->k_pool +"),
    "q row of the kv head": ("P->q + ((int64_t)b * P->Hq + h) * P->D",
                             "P->q + ((int64_t)b * P->Hq + h / (P->Hq / P->Hkv)) * P->D"),
    "last token dropped": ("return attend_prefix(P, b, h, P->seq_lens[b], qrow, out);",
                           "return attend_prefix(P, b, h, P->seq_lens[b] > 1 ? P->seq_lens[b] - 1 : "
                           "P->seq_lens[b], qrow, out);"),
    "causal limit off by one": ("int32_t n = P->seq_lens[b] - j->q_len + 1 + qi;",
                                "int32_t n = P->seq_lens[b] - j->q_len + qi;"),
    "every query uses the first q row": ("const uint16_t* qrow = P->q + i * P->D;",
                                         "const uint16_t* qrow = P->q + (i - (int64_t)qi * P->Hq) * P->D;"),
    "slot from block index": ("return blk * P->blk_stride + (int64_t)slot * P->tok_stride",
                              "return blk * P->blk_stride + (int64_t)(slot / 2) * P->tok_stride"),
    "bf16 widened as low half": ("uint32_t u = ((uint32_t)bits) << 16;", "uint32_t u = ((uint32_t)bits) << 15;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    with open(oracle.SOURCE) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation anchor missing: {old!r}"
    mutated = src.replace(old, new, 1)
    path = tmp_path / "pda_oracle.c"
    path.write_text(mutated)
    header = os.path.join(os.path.dirname(oracle.SOURCE), "pda_oracle.h")
    (tmp_path / "pda_oracle.h").write_text(open(header).read())
    lib = oracle.build(str(path), str(tmp_path / "libmut.so"))
    failed = oracle_pins.failing_pins(oracle.Oracle(lib))
    assert failed, f"mutant '{name}' passed every pin"
