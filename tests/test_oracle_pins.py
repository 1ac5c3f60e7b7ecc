"""The fp64 oracle against its pins (CPU only)."""
import numpy as np
import pytest

import oracle
from tests import oracle_pins


def _attn(q, k, v, scale, causal, rows=None):
    return oracle.attention(q, k, v, scale, causal, rows=rows)


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(_attn)


def test_oracle_e4m3_pins():
    def attn8(q, k, v, scale, ds, causal, rows=None):
        return oracle.attention_e4m3(q, k, v, scale, ds, causal, rows=rows)
    oracle_pins.pin_e4m3_decode(oracle.e4m3_decode)
    oracle_pins.pin_e4m3_sdpa_library(attn8)
    oracle_pins.pin_e4m3_matches_bf16_path(attn8, _attn)


def test_oracle_block_mask_pins():
    def attnm(q, k, v, scale, mask, causal, rows=None):
        return oracle.attention_masked(q, k, v, scale, mask, causal, rows=rows)
    oracle_pins.pin_block_mask_library(attnm)
    oracle_pins.pin_block_mask_all_ones(attnm, _attn)


def _bwd(q, k, v, dout, scale, causal, kv_heads=None):
    return oracle.attention_bwd(q, k, v, dout, scale, causal, kv_heads=kv_heads)


def test_oracle_bwd_finite_differences():
    oracle_pins.pin_bwd_finite_differences(_bwd, oracle.attention_f64)


@pytest.mark.parametrize("pin", oracle_pins.BWD_PINS, ids=lambda p: p.__name__)
def test_oracle_bwd_pin(pin):
    pin(_bwd)


def _bwdm(q, k, v, dout, scale, causal, mask, kv_heads=None):
    return oracle.attention_bwd(q, k, v, dout, scale, causal, kv_heads=kv_heads, block_mask=mask)


def test_oracle_bwd_masked_pins():
    oracle_pins.pin_bwd_masked_library(_bwdm)
    oracle_pins.pin_bwd_masked_all_ones(_bwdm, _bwd)


def test_oracle_bwd_thread_count_does_not_change_bits():
    from causal_scaled_dot_gb300.inputs import gaussian_bf16, qkv_bf16
    q, k, v = qkv_bf16(1, 4, 2, 50, 8, seed=10)
    do = gaussian_bf16((1, 4, 50, 8), 10, 3)
    a = oracle.attention_bwd(q, k, v, do, 0.3, True, nthreads=1)
    b = oracle.attention_bwd(q, k, v, do, 0.3, True, nthreads=6)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))


def test_test_side_philox_gives_the_published_known_answers():
    oracle_pins.pin_test_generator_known_answers()


def test_oracle_philox_known_answers():
    oracle_pins.pin_philox_known_answers(oracle.philox4x32)


def test_oracle_philox_pin():
    oracle_pins.pin_philox_library(oracle.philox4x32)


def test_oracle_rejects_offsets_past_32_bits():
    from causal_scaled_dot_gb300.inputs import qkv_bf16
    q, k, v = qkv_bf16(1, 1, 1, 20, 8, seed=11)
    oracle.attention_dropout(q, k, v, 0.3, 10, 1, 2**32 - 1, True)
    with pytest.raises(ValueError):
        oracle.attention_dropout(q, k, v, 0.3, 10, 1, 2**32, True)


def _attnd(q, k, v, scale, p8, seed, offset, causal, rows=None):
    return oracle.attention_dropout(q, k, v, scale, p8, seed, offset, causal, rows=rows)


@pytest.mark.parametrize("pin", oracle_pins.DROPOUT_PINS, ids=lambda p: p.__name__)
def test_oracle_dropout_pin(pin):
    pin(_attnd, _attn)


@pytest.mark.parametrize("pin", oracle_pins.PROJ_PINS, ids=lambda p: p.__name__)
def test_oracle_proj_pin(pin):
    pin(oracle.out_proj)


def test_proj_pins_catch_planted_mistakes():
    """Plausible slips in the projection's index mapping or bias: some pin fails for each."""
    import numpy as _np

    def wide(x):
        x = _np.asarray(x)
        return (x.astype(_np.uint32) << _np.uint32(16)).view(_np.float32).astype(_np.float64) \
            if x.dtype == _np.uint16 else x.astype(_np.float64)

    def heads_major(o, w, bias=None):      # k = d*H + h instead of h*D + d
        O, W = wide(o), wide(w)
        B, H, S, D = O.shape
        Y = O.transpose(0, 2, 3, 1).reshape(B, S, H * D) @ W.T
        return Y + (0 if bias is None else _np.asarray(bias))

    def w_transposed(o, w, bias=None):     # W read as [H*D, E] memory
        O, W = wide(o), wide(w)
        B, H, S, D = O.shape
        Wt = W.reshape(-1).reshape(W.shape[1], W.shape[0]).T
        Y = O.transpose(0, 2, 1, 3).reshape(B, S, H * D) @ Wt.T
        return Y + (0 if bias is None else _np.asarray(bias))

    def bias_dropped(o, w, bias=None):
        return oracle.out_proj(o, w, None)

    def seq_head_swapped(o, w, bias=None):  # O read as [B, S, H, D]
        O, W = wide(o), wide(w)
        B, H, S, D = O.shape
        Y = O.reshape(B, S, H * D) @ W.T
        return Y + (0 if bias is None else _np.asarray(bias))

    for mutant in (heads_major, w_transposed, bias_dropped, seq_head_swapped):
        caught = 0
        for pin in oracle_pins.PROJ_PINS:
            try:
                pin(mutant)
            except (AssertionError, ValueError):
                caught += 1
        assert caught, mutant.__name__


def test_rows_subset_matches_full():
    """The row-selection entry computes exactly the rows of the full call."""
    from causal_scaled_dot_gb300.inputs import qkv_bf16
    q, k, v = qkv_bf16(2, 4, 2, 33, 16, seed=7)
    O, L = oracle.attention(q, k, v, 0.25, True)
    rows = np.array([0, 1, 32, 33, 100, 2 * 4 * 33 - 1], dtype=np.int64)
    Or, Lr = oracle.attention(q, k, v, 0.25, True, rows=rows)
    assert np.array_equal(Or, O.reshape(-1, 16)[rows])
    assert np.array_equal(Lr, L.reshape(-1)[rows])


def test_thread_count_does_not_change_bits():
    from causal_scaled_dot_gb300.inputs import qkv_bf16
    q, k, v = qkv_bf16(1, 2, 2, 70, 8, seed=8)
    a = oracle.attention(q, k, v, 0.3, True, nthreads=1)
    b = oracle.attention(q, k, v, 0.3, True, nthreads=5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_oracle_rejects_bad_arguments():
    from causal_scaled_dot_gb300.inputs import qkv_bf16
    q, k, v = qkv_bf16(1, 3, 2, 8, 8, seed=9)  # Hq % Hkv != 0
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, 0.3, True)
    q, k, v = qkv_bf16(1, 2, 2, 8, 8, seed=9)
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, 0.3, True, rows=np.array([16], np.int64))
    with pytest.raises(TypeError):
        oracle.attention(q.astype(np.float32), k, v, 0.3, True)


def test_oracle_snapshot_small_workload():
    """Seeded inputs + oracle reproduce the committed snapshot on this host."""
    import os
    from causal_scaled_dot_gb300.inputs import qkv_bf16
    from causal_scaled_dot_gb300.workloads import SMALL as w
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_small_rows.txt")
    rows, lse_ref, out_ref = [], [], []
    for line in open(path):
        if line.startswith("#"):
            continue
        f = line.split()
        rows.append(int(f[0])); lse_ref.append(float(f[1])); out_ref.append([float(x) for x in f[2:]])
    q, k, v = qkv_bf16(w.B, w.Hq, w.Hkv, w.S, w.D, seed=w.seed, sigma=w.sigma)
    out, lse = oracle.attention(q, k, v, w.scale, w.causal, rows=np.array(rows, np.int64))
    out_ref = np.array(out_ref)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(out[:, :out_ref.shape[1]], out_ref, rtol=0, atol=1e-12)


def _attnk(q, k, v, scale, bits, causal, block_mask=None, rows=None):
    return oracle.attention_keep(q, k, v, scale, bits, causal, block_mask=block_mask, rows=rows)


@pytest.mark.parametrize("pin", oracle_pins.KEEP_PINS, ids=lambda p: p.__name__)
def test_oracle_keep_pin(pin):
    pin(_attnk)


def test_oracle_keep_equals_block_mask():
    def attnm(q, k, v, scale, mask, causal, rows=None):
        return oracle.attention_masked(q, k, v, scale, mask, causal, rows=rows)
    oracle_pins.pin_keep_equals_block_mask(_attnk, attnm)


def _bwdk(q, k, v, dout, scale, causal, bits, kv_heads=None):
    return oracle.attention_bwd(q, k, v, dout, scale, causal, kv_heads=kv_heads, keep_bits=bits)


@pytest.mark.parametrize("pin", oracle_pins.BWD_KEEP_PINS, ids=lambda p: p.__name__)
def test_oracle_bwd_keep_pin(pin):
    pin(_bwdk)


def _bwdd(q, k, v, dout, scale, causal, dropout, kv_heads=None):
    return oracle.attention_bwd(q, k, v, dout, scale, causal, kv_heads=kv_heads, dropout=dropout)


@pytest.mark.parametrize("pin", oracle_pins.BWD_DROPOUT_PINS, ids=lambda p: p.__name__)
def test_oracle_bwd_dropout_pin(pin):
    pin(_bwdd)


def _attnx(q, k, v, scale, causal, descales=None, block_mask=None, keep_bits=None, dropout=None):
    return oracle.attention_ex(q, k, v, scale, causal, descales=descales, block_mask=block_mask,
                               keep_bits=keep_bits, dropout=dropout)


@pytest.mark.parametrize("pin", oracle_pins.COMBO_PINS, ids=lambda p: p.__name__)
def test_oracle_combo_pin(pin):
    pin(_attnx)


def _bwdx(q, k, v, dout, scale, causal, block_mask, keep_bits, dropout):
    return oracle.attention_bwd(q, k, v, dout, scale, causal, block_mask=block_mask, keep_bits=keep_bits,
                                dropout=dropout)


@pytest.mark.parametrize("pin", oracle_pins.BWD_COMBO_PINS, ids=lambda p: p.__name__)
def test_oracle_bwd_combo_pin(pin):
    pin(_bwdx)
