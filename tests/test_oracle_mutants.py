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
    "key_operand_transposed": ("elem(J, 1, kb + j * D + d)", "elem(J, 1, kb + d * S + j)"),
    "gqa_interleaved": ("const int64_t hkv = hq / G;", "const int64_t hkv = hq % J->Hkv;"),
    "lse_without_max": ("*lse_out = m + log(l);", "*lse_out = log(l);"),
    "no_max_subtraction": ("s[j] = exp(s[j] - m);", "s[j] = exp(s[j]);"),
    "exp_sign_flipped": ("s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    "normalisation_dropped": ("for (int64_t j = 0; j < S; ++j) s[j] = s[j] / l;", ""),
    "value_row_is_query_row": ("elem(J, 2, vb + j * D + d)", "elem(J, 2, vb + i * D + d)"),
    "batch_offset_dropped": ("const int64_t kb = ((b * J->Hkv + hkv) * S) * (int64_t)D;",
                             "const int64_t kb = ((hkv) * S) * (int64_t)D;"),
    "query_row_offset_wrong": ("const int64_t qi = (bh * S + i) * (int64_t)D;",
                               "const int64_t qi = (bh * S) * (int64_t)D;"),
    "lse_log2": ("*lse_out = m + log(l);", "*lse_out = m + log2(l);"),
    "e4m3_exponent_bias": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    "e4m3_subnormal_scale": ("ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    "e4m3_descale_ignored": ("e4m3_bits_to_double(((const uint8_t *)J->t[which])[idx]) * J->descale[which]",
                             "e4m3_bits_to_double(((const uint8_t *)J->t[which])[idx])"),
    "e4m3_descale_swapped": ("J->descale[which]", "J->descale[2 - which]"),
    "block_mask_transposed": ("if (mrow[j / 128] == 0) s[j] = -INFINITY;",
                              "if (J->block_mask[(j / 128) * ((S + 127) / 128) + i / 128] == 0) s[j] = -INFINITY;"),
    "block_mask_heads_ignored": ("(J->mask_heads == 1 ? 0 : hq)", "(0)"),
    "block_mask_ignored": ("if (J->block_mask) {", "if (0) {"),
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

    def attn8(q, k, v, scale, ds, causal, rows=None):
        return oracle.attention_e4m3(q, k, v, scale, ds, causal, rows=rows, lib=lib)

    def attnm(q, k, v, scale, mask, causal, rows=None):
        return oracle.attention_masked(q, k, v, scale, mask, causal, rows=rows, lib=lib)

    checks = [(p.__name__, lambda p=p: p(attn)) for p in oracle_pins.ALL_PINS] + [
        ("pin_e4m3_decode", lambda: oracle_pins.pin_e4m3_decode(
            lambda c: oracle.e4m3_decode(c, lib=lib))),
        ("pin_e4m3_sdpa_library", lambda: oracle_pins.pin_e4m3_sdpa_library(attn8)),
        ("pin_e4m3_matches_bf16_path", lambda: oracle_pins.pin_e4m3_matches_bf16_path(attn8, attn)),
        ("pin_block_mask_library", lambda: oracle_pins.pin_block_mask_library(attnm)),
        ("pin_block_mask_all_ones", lambda: oracle_pins.pin_block_mask_all_ones(attnm, attn)),
    ]
    caught = []
    for pin_name, run in checks:
        try:
            run()
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin_name)
    assert caught, f"no pin caught mutant {name}"
