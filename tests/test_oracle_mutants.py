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
    "dropout_keep_flipped": ("return byte >= J->dropout_p8;", "return byte < J->dropout_p8;"),
    "dropout_byte_order": ("(out[(j % 16) / 4] >> (8 * (j % 4)))", "(out[(j % 16) % 4] >> (8 * ((j % 16) / 4)))"),
    "dropout_counter_swapped": ("{(uint32_t)(j / 16), (uint32_t)i, (uint32_t)bh,",
                                "{(uint32_t)i, (uint32_t)(j / 16), (uint32_t)bh,"),
    "dropout_offset_dropped": ("(uint32_t)bh, (uint32_t)J->dropout_offset};", "(uint32_t)bh, 0u};"),
    "dropout_key_words_swapped": ("{(uint32_t)(J->dropout_seed & 0xFFFFFFFFu), (uint32_t)(J->dropout_seed >> 32)}",
                                  "{(uint32_t)(J->dropout_seed >> 32), (uint32_t)(J->dropout_seed & 0xFFFFFFFFu)}"),
    "dropout_unscaled": ("s[j] = dropout_keeps(J, r / S, i, j) ? s[j] * keep_scale : 0.0;",
                         "s[j] = dropout_keeps(J, r / S, i, j) ? s[j] : 0.0;"),
    "philox_weyl_swapped": ("k0 += W0;\n        k1 += W1;", "k0 += W1;\n        k1 += W0;"),
    "philox_round_outputs_swapped": ("x1 = lo1;", "x1 = lo0;"),
    "bwd_delta_not_subtracted": ("ds[j] = p[j] * (dP[j] - delta);", "ds[j] = p[j] * dP[j];"),
    "bwd_delta_unweighted": ("delta += p[j] * dP[j];", "delta += dP[j];"),
    "bwd_dq_scale_dropped": ("for (int d = 0; d < D; ++d) dq[d] *= J->scale;", ""),
    "bwd_dk_scale_dropped": ("for (int d = 0; d < D; ++d) dk[d] *= J->scale;", ""),
    "bwd_dv_uses_score_gradient": ("dv[d] += wij * elem(J, 3, qo + d);",
                                   "dv[d] += dsij * elem(J, 3, qo + d);"),
    "bwd_dk_uses_weights": ("dk[d] += dsij * elem(J, 0, qo + d);",
                            "dk[d] += pij * elem(J, 0, qo + d);"),
    "bwd_dq_uses_values": ("dq[d] += ds[j] * elem(J, 1, kvb + j * D + d);",
                           "dq[d] += ds[j] * elem(J, 2, kvb + j * D + d);"),
    "bwd_dp_uses_keys": ("dP[j] += elem(J, 3, qo + d) * elem(J, 2, kvb + j * D + d);",
                         "dP[j] += elem(J, 3, qo + d) * elem(J, 1, kvb + j * D + d);"),
    "bwd_group_interleaved": ("const int64_t hq = W->hkv * W->G + g;",
                              "const int64_t hq = W->hkv + g * J->Hkv;"),
    "bwd_dkdv_first_head_only": ("for (int64_t g = 0; g < W->G; ++g) {",
                                 "for (int64_t g = 0; g < 1; ++g) {"),
    "keep_bit_order_reversed": ("if (((krow[j / 8] >> (j % 8)) & 1) == 0)",
                                "if (((krow[j / 8] >> (7 - j % 8)) & 1) == 0)"),
    "keep_row_stride_unpadded": ("const int64_t row_bytes = 16 * ((S + 127) / 128);",
                                 "const int64_t row_bytes = (S + 7) / 8;"),
    "keep_heads_ignored": ("(J->keep_heads == 1 ? 0 : hq)", "(0)"),
    "keep_ignored": ("if (J->keep_bits) {", "if (0) {"),
    "bwd_dropout_dv_undropped": ("wij = dropout_keeps(J, bh, i, j) ? pij * (256.0 / (256.0 - (double)J->dropout_p8)) : 0.0;",
                                 "wij = pij;"),
    "ex_descales_ignored": ("format == FMT_E4M3 ? ds : one", "one"),
    "ex_mask_heads_collapsed": ("causal, block_mask, block_mask ? mask_heads : 1, keep_bits,\n",
                                "causal, block_mask, 1, keep_bits,\n"),
    "ex_dropout_dropped": ("keep_bits ? keep_heads : 1, p8, seed, offset, rows,",
                           "keep_bits ? keep_heads : 1, 0, seed, offset, rows,"),
    "ex_bwd_keep_dropped": ("keep_bits, keep_bits ? keep_heads : 1, p8, seed, offset,",
                            "NULL, 1, p8, seed, offset,"),
    "ex_bwd_seed_offset_swapped": ("keep_heads : 1, p8, seed, offset,\n                   kv_heads",
                                   "keep_heads : 1, p8, offset, seed,\n                   kv_heads"),
    "dropout_counter_batch_dropped": ("s[j] = dropout_keeps(J, r / S, i, j) ? s[j] * keep_scale : 0.0;",
                                      "s[j] = dropout_keeps(J, (r / S) % J->Hq, i, j) ? s[j] * keep_scale : 0.0;"),
    "bwd_dropout_counter_batch_dropped": ("wij = dropout_keeps(J, bh, i, j) ?",
                                          "wij = dropout_keeps(J, bh % J->Hq, i, j) ?"),
    "bwd_dropout_dp_unscaled": ("if (p[j] != 0.0) dP[j] = dropout_keeps(J, bh, i, j) ? dP[j] * keep_scale : 0.0;",
                                "if (p[j] != 0.0) dP[j] = dropout_keeps(J, bh, i, j) ? dP[j] : 0.0;"),
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

    def attnk(q, k, v, scale, bits, causal, block_mask=None, rows=None):
        return oracle.attention_keep(q, k, v, scale, bits, causal, block_mask=block_mask, rows=rows,
                                     lib=lib)

    def attnd(q, k, v, scale, p8, seed, offset, causal, rows=None):
        return oracle.attention_dropout(q, k, v, scale, p8, seed, offset, causal, rows=rows, lib=lib)

    def bwd(q, k, v, dout, scale, causal, kv_heads=None):
        return oracle.attention_bwd(q, k, v, dout, scale, causal, kv_heads=kv_heads, lib=lib)

    def fwd64(q, k, v, scale, causal):
        return oracle.attention_f64(q, k, v, scale, causal, nthreads=1, lib=lib)

    def attnx(q, k, v, scale, causal, descales=None, block_mask=None, keep_bits=None, dropout=None):
        return oracle.attention_ex(q, k, v, scale, causal, descales=descales, block_mask=block_mask,
                                   keep_bits=keep_bits, dropout=dropout, lib=lib)

    def bwdx(q, k, v, dout, scale, causal, block_mask, keep_bits, dropout):
        return oracle.attention_bwd(q, k, v, dout, scale, causal, block_mask=block_mask, keep_bits=keep_bits,
                                    dropout=dropout, lib=lib)

    checks = [(p.__name__, lambda p=p: p(attn)) for p in oracle_pins.ALL_PINS] + [
        ("pin_e4m3_decode", lambda: oracle_pins.pin_e4m3_decode(
            lambda c: oracle.e4m3_decode(c, lib=lib))),
        ("pin_e4m3_sdpa_library", lambda: oracle_pins.pin_e4m3_sdpa_library(attn8)),
        ("pin_e4m3_matches_bf16_path", lambda: oracle_pins.pin_e4m3_matches_bf16_path(attn8, attn)),
        ("pin_block_mask_library", lambda: oracle_pins.pin_block_mask_library(attnm)),
        ("pin_block_mask_all_ones", lambda: oracle_pins.pin_block_mask_all_ones(attnm, attn)),
        ("pin_bwd_finite_differences", lambda: oracle_pins.pin_bwd_finite_differences(bwd, fwd64)),
    ] + [(p.__name__, lambda p=p: p(bwd)) for p in oracle_pins.BWD_PINS] + [
        ("pin_philox_known_answers", lambda: oracle_pins.pin_philox_known_answers(
            lambda c, k: oracle.philox4x32(c, k, lib=lib))),
    ] + [(p.__name__, lambda p=p: p(attnd, attn)) for p in oracle_pins.DROPOUT_PINS] + [
        ("pin_bwd_masked_library", lambda: oracle_pins.pin_bwd_masked_library(
            lambda q, k, v, d, sc, c, m: oracle.attention_bwd(q, k, v, d, sc, c, block_mask=m, lib=lib))),
    ] + [(p.__name__, lambda p=p: p(attnk)) for p in oracle_pins.KEEP_PINS] + [
        ("pin_keep_equals_block_mask", lambda: oracle_pins.pin_keep_equals_block_mask(attnk, attnm)),
        ("pin_bwd_keep_library", lambda: oracle_pins.pin_bwd_keep_library(
            lambda q, k, v, d, sc, c, b: oracle.attention_bwd(q, k, v, d, sc, c, keep_bits=b, lib=lib))),
        ("pin_bwd_dropout_autograd", lambda: oracle_pins.pin_bwd_dropout_autograd(
            lambda q, k, v, d, sc, c, dr: oracle.attention_bwd(q, k, v, d, sc, c, dropout=dr, lib=lib))),
    ] + [(p.__name__, lambda p=p: p(attnx)) for p in oracle_pins.COMBO_PINS] + [
        (p.__name__, lambda p=p: p(bwdx)) for p in oracle_pins.BWD_COMBO_PINS]
    caught = []
    for pin_name, run in checks:
        try:
            run()
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin_name)
    assert caught, f"no pin caught mutant {name}"
