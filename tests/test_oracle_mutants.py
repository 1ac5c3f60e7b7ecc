"""Plant mistakes in copies of the oracle's C source; some pin must catch each.

Each mutant is a plausible slip (a dropped term, a wrong sign or index, a
transposed operand, a wrong mask or head mapping).  The copy is compiled into
a temporary directory; the oracle itself is never modified.
"""
import os

import pytest

import oracle
from tests import oracle_pins

MUTANTS = {
    "mask_keeps_diagonal_out": ("for (int64_t j = i + 1; j < S; ++j) s[j] = -INFINITY;",
                                "for (int64_t j = i; j < S; ++j) s[j] = -INFINITY;"),
    "mask_off_by_one_late": ("for (int64_t j = i + 1; j < S; ++j) s[j] = -INFINITY;",
                             "for (int64_t j = i + 2; j < S; ++j) s[j] = -INFINITY;"),
    "scale_dropped": ("s[j] = s[j] * J->scale;", "s[j] = s[j];"),
    "key_operand_transposed": ("bf16_bits_to_double(kb[j * D + d])",
                               "bf16_bits_to_double(kb[d * S + j])"),
    "gqa_interleaved": ("const int64_t hkv = hq / G;", "const int64_t hkv = hq % J->Hkv;"),
    "lse_without_max": ("*lse_out = m + log(l);", "*lse_out = log(l);"),
    "no_max_subtraction": ("s[j] = exp(s[j] - m);", "s[j] = exp(s[j]);"),
    "exp_sign_flipped": ("s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    "normalisation_dropped": ("for (int64_t j = 0; j < S; ++j) s[j] = s[j] / l;", ""),
    "value_row_is_query_row": ("bf16_bits_to_double(vb[j * D + d])",
                               "bf16_bits_to_double(vb[i * D + d])"),
    "batch_offset_dropped": ("const uint16_t *kb = J->k + ((b * J->Hkv + hkv) * S) * (int64_t)D;",
                             "const uint16_t *kb = J->k + ((hkv) * S) * (int64_t)D;"),
    "query_row_offset_wrong": ("const uint16_t *qi = J->q + (bh * S + i) * (int64_t)D;",
                               "const uint16_t *qi = J->q + (bh * S) * (int64_t)D;"),
    "lse_log2": ("*lse_out = m + log(l);", "*lse_out = m + log2(l);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_some_pin_catches_mutant(name, tmp_path):
    src = open(oracle.SOURCE).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib_path = oracle.compile_oracle(str(mutated), str(tmp_path / "libmutant.so"))
    lib = oracle._bind(__import__("ctypes").CDLL(lib_path))

    def attn(q, k, v, scale, causal, rows=None):
        return oracle.attention(q, k, v, scale, causal, rows=rows, lib=lib)

    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(attn)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name}"
