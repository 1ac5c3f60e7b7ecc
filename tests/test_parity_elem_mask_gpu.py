"""GPU parity of the element-masked forward (attn_fwd_elem_masked) against the
oracle: random keep bits (shared and per head), local windows with and without
the matching block mask, rows that see no key, the all-ones mask against the
unmasked kernel, and sampled rows of the full-size workloads."""
import math

import numpy as np
import pytest

import oracle
from causal_scaled_dot_gb300.inputs import (block_mask_of_keep_bits, qkv_bf16, random_block_mask,
                                            random_keep_bits, window_keep_bits)
from causal_scaled_dot_gb300.workloads import WORKLOADS
from tests.gpu_util import compare_masked, run_gpu, run_gpu_elem_masked, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _check(B, Hq, Hkv, S, D, causal, bits, seed, block_mask=None, rows=None, sigma=1.0):
    q, k, v = qkv_bf16(B, Hq, Hkv, S, D, seed=seed, sigma=sigma)
    scale = 1.0 / math.sqrt(D)
    o, l = run_gpu_elem_masked(q, k, v, scale, causal, bits, block_mask)
    ro, rl = oracle.attention_keep(q, k, v, scale, bits, causal, block_mask=block_mask, rows=rows)
    if rows is not None:
        o, l = o.reshape(-1, D)[rows], l.reshape(-1)[rows]
    label = f"elem mask B{B} Hq{Hq} Hkv{Hkv} S{S} D{D} causal={causal} Hm={bits.shape[0]}"
    return compare_masked(o, ro, l, rl, label), (o, l)


@pytest.mark.parametrize("S", [129, 300, 1000])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("density", [0.1, 0.5, 0.9])
def test_elem_mask_random(S, D, causal, density):
    Hq = 4
    per_head = (S + D) % 2 == 0
    bits = random_keep_bits(Hq if per_head else 1, S, density, seed=S + D + int(100 * density))
    print(_check(2, Hq, 2, S, D, causal, bits, seed=6100 + S + D)[0])


def test_elem_mask_rows_without_keys():
    """Query rows 3 and 200 of head 1 keep nothing; a whole 32-row warp of head 0
    keeps nothing; every other row keeps its diagonal at least."""
    S, Hq = 300, 2
    from causal_scaled_dot_gb300.inputs import pack_keep_bits
    rng = np.random.default_rng(5)
    keep = rng.random((Hq, S, S)) < 0.3
    keep[:, np.arange(S), np.arange(S)] = True
    keep[1, 3, :] = False
    keep[1, 200, :] = False
    keep[0, 32:64, :] = False
    stats, (o, l) = _check(1, Hq, Hq, S, 128, True, pack_keep_bits(keep), seed=6200)
    assert stats["empty_rows"] == 34


@pytest.mark.parametrize("window", [1, 100, 256, 700])
def test_elem_mask_local_window_with_and_without_block_mask(window):
    """A sliding window: with the derived block mask (dropped blocks skipped) and
    without it (every causal block computed) the results agree bit for bit."""
    S, D = 1000, 128
    bits = window_keep_bits(S, window)
    bm = block_mask_of_keep_bits(bits, S)
    _, (o1, l1) = _check(1, 4, 2, S, D, True, bits, seed=6300 + window)
    _, (o2, l2) = _check(1, 4, 2, S, D, True, bits, seed=6300 + window, block_mask=bm)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_elem_mask_with_random_block_mask():
    S, Hq = 700, 4
    bits = random_keep_bits(Hq, S, 0.6, seed=64)
    bm = random_block_mask(Hq, S, 0.6, seed=65)
    print(_check(2, Hq, 2, S, 64, True, bits, seed=6400, block_mask=bm)[0])
    print(_check(2, Hq, 2, S, 128, False, bits, seed=6401, block_mask=bm)[0])


def test_elem_mask_all_ones_equals_unmasked():
    B, Hq, Hkv, S, D = 2, 4, 2, 700, 128
    q, k, v = qkv_bf16(B, Hq, Hkv, S, D, seed=6500)
    ones = np.full((1, S, 16 * ((S + 127) // 128)), 0xFF, np.uint8)
    for causal in (True, False):
        a = run_gpu_elem_masked(q, k, v, 0.088, causal, ones)
        b = run_gpu(q, k, v, 0.088, causal)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("w", WORKLOADS[1:], ids=lambda w: w.name)
def test_elem_mask_full_size_sampled_rows(w):
    """The launch the benchmark times: a 1024-key local window with its block mask."""
    bits = window_keep_bits(w.S, 1024)
    bm = block_mask_of_keep_bits(bits, w.S)
    rows = sample_rows(w.B, w.Hq, w.S, n_random=128, seed=w.seed)
    print(w.name, _check(w.B, w.Hq, w.Hkv, w.S, w.D, True, bits, seed=w.seed, block_mask=bm, rows=rows,
                         sigma=w.sigma)[0])
