"""GPU parity of the block-masked entry point against the fp64 oracle: random
block masks (shared and per head), causal and not, GQA, ragged tails, blocks
dropped so that whole query tiles see no key, and the all-ones mask, which
must reproduce the unmasked call bit for bit."""
import math

import numpy as np
import pytest

import oracle
from causal_scaled_dot_gb300.inputs import qkv_bf16, random_block_mask
from causal_scaled_dot_gb300.workloads import WORKLOADS
from tests.gpu_util import compare_masked, run_gpu, run_gpu_masked, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _check(B, Hq, Hkv, S, D, causal, mask, seed, rows=None, sigma=1.0):
    q, k, v = qkv_bf16(B, Hq, Hkv, S, D, seed=seed, sigma=sigma)
    scale = 1.0 / math.sqrt(D)
    o, l = run_gpu_masked(q, k, v, scale, causal, mask)
    o_ref, l_ref = oracle.attention_masked(q, k, v, scale, mask, causal, rows=rows)
    if rows is not None:
        o, l = o.reshape(-1, D)[rows], l.reshape(-1)[rows]
    return compare_masked(o, o_ref, l, l_ref,
                          f"masked B{B} Hq{Hq} Hkv{Hkv} S{S} D{D} causal={causal} Hm={mask.shape[0]}")


@pytest.mark.parametrize("S", [1, 129, 300, 1000])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("per_head", [False, True])
def test_random_masks(S, D, causal, per_head):
    Hq = 4
    mask = random_block_mask(Hq if per_head else 1, S, 0.6, seed=S + D)
    print(_check(2, Hq, 2, S, D, causal, mask, seed=1400 + S + D))


@pytest.mark.parametrize("density", [0.1, 0.3, 0.9])
def test_mask_densities_gqa(density):
    S, Hq = 1500, 8
    mask = random_block_mask(Hq, S, density, seed=int(density * 100))
    print(_check(1, Hq, 2, S, 128, True, mask, seed=1500))


def test_all_ones_mask_equals_unmasked_bitwise():
    for causal in (True, False):
        B, Hq, Hkv, S, D = 2, 4, 2, 700, 128
        q, k, v = qkv_bf16(B, Hq, Hkv, S, D, seed=1600)
        scale = 1.0 / math.sqrt(D)
        nt = (S + 127) // 128
        o_m, l_m = run_gpu_masked(q, k, v, scale, causal, np.ones((1, nt, nt), np.uint8))
        o_u, l_u, _ = run_gpu(q, k, v, scale, causal)
        assert np.array_equal(o_m, o_u) and np.array_equal(l_m, l_u)


def test_empty_query_tiles_give_zero_and_minus_inf():
    """Query tile 0 of head 0 keeps no block, tile 2 of every head keeps none
    either: those rows see no key at all."""
    S, Hq = 600, 2
    nt = (S + 127) // 128
    mask = np.ones((Hq, nt, nt), np.uint8)
    mask[0, 0, :] = 0
    mask[:, 2, :] = 0
    st = _check(1, Hq, 1, S, 128, True, mask, seed=1700)
    assert st["empty_rows"] == 128 + 2 * 128


def test_diagonal_block_dropped_under_causal():
    """Dropping the diagonal block leaves each query only the keys of earlier
    tiles; tile 0 then sees nothing."""
    S = 900
    nt = (S + 127) // 128
    mask = np.ones((1, nt, nt), np.uint8)
    mask[0, np.arange(nt), np.arange(nt)] = 0
    st = _check(1, 2, 2, S, 128, True, mask, seed=1800)
    assert st["empty_rows"] == 2 * 128


def test_local_band_mask():
    """A sliding window of one tile: the diagonal block and the one before it."""
    S = 2000
    nt = (S + 127) // 128
    i = np.arange(nt)
    mask = ((i[:, None] - i[None, :] >= 0) & (i[:, None] - i[None, :] <= 1)).astype(np.uint8)
    _check(2, 4, 4, S, 128, True, mask[None], seed=1900)


def test_all_zero_mask():
    S = 256
    mask = np.zeros((1, 2, 2), np.uint8)
    st = _check(1, 2, 1, S, 64, False, mask, seed=2000)
    assert st["empty_rows"] == 2 * S


@pytest.mark.parametrize("w", WORKLOADS[1:], ids=lambda w: w.name)
def test_full_size_workloads_masked_sampled_rows(w):
    mask = random_block_mask(w.Hq, w.S, 0.5, seed=w.seed)
    rows = sample_rows(w.B, w.Hq, w.S, n_random=256, seed=w.seed)
    print(w.name, _check(w.B, w.Hq, w.Hkv, w.S, w.D, True, mask, seed=w.seed, rows=rows,
                         sigma=w.sigma))


@pytest.mark.parametrize("density", [0.0, 0.05])
def test_sparse_masks_many_empty_units(density):
    """Long runs of query tiles that keep no key tile, in every CTA."""
    S, Hq = 2048, 32
    mask = random_block_mask(Hq, S, density, seed=2100)
    q, k, v = qkv_bf16(1, Hq, Hq, S, 128, seed=2100)
    o, l = run_gpu_masked(q, k, v, 128 ** -0.5, True, mask)
    if density == 0.0:
        assert not o.any() and np.all(np.isneginf(l))
        return
    rows = sample_rows(1, Hq, S, n_random=512, seed=2100)
    o_ref, l_ref = oracle.attention_masked(q, k, v, 128 ** -0.5, mask, True, rows=rows)
    print(compare_masked(o.reshape(-1, 128)[rows], o_ref, l.reshape(-1)[rows], l_ref, "sparse"))
