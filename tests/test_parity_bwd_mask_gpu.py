"""GPU parity of the block-masked backward (attn_bwd_block_masked after
attn_fwd_block_masked) against the oracle's block-masked gradients, with the
tolerances of the unmasked backward (tests/gpu_util).  Includes query tiles
that keep no key tile (their dQ is exactly 0) and key tiles that no query tile
keeps (their dK, dV are exactly 0)."""
import math

import numpy as np
import pytest

import oracle
from causal_scaled_dot_gb300.inputs import gaussian_bf16, qkv_bf16, random_block_mask
from causal_scaled_dot_gb300.workloads import WORKLOADS
from tests.gpu_util import compare_grad, run_gpu_bwd, run_gpu_bwd_masked

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _check(B, Hq, Hkv, S, D, causal, mask, seed, kv_heads=None, sigma=1.0):
    q, k, v = qkv_bf16(B, Hq, Hkv, S, D, seed=seed, sigma=sigma)
    do = gaussian_bf16((B, Hq, S, D), seed, 3)
    scale = 1.0 / math.sqrt(D)
    _, _, dq, dk, dv, _ = run_gpu_bwd_masked(q, k, v, do, scale, causal, mask)
    rq, rk, rv, _ = oracle.attention_bwd(q, k, v, do, scale, causal, kv_heads=kv_heads, block_mask=mask)
    G = Hq // Hkv
    if kv_heads is not None:
        sel = np.asarray(kv_heads)
        dq = dq.reshape(B * Hkv, G, S, D)[sel]
        dk = dk.reshape(B * Hkv, S, D)[sel]
        dv = dv.reshape(B * Hkv, S, D)[sel]
    label = f"masked bwd B{B} Hq{Hq} Hkv{Hkv} S{S} D{D} causal={causal} Hm={mask.shape[0]}"
    return {"dq": compare_grad(dq, rq, label + " dQ"), "dk": compare_grad(dk, rk, label + " dK"),
            "dv": compare_grad(dv, rv, label + " dV")}, (dq, dk, dv, rq, rk, rv)


@pytest.mark.parametrize("S", [129, 300, 1000])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("per_head", [False, True])
def test_masked_bwd_random_masks(S, D, causal, per_head):
    Hq = 4
    mask = random_block_mask(Hq if per_head else 1, S, 0.6, seed=S + D + 7)
    print(_check(2, Hq, 2, S, D, causal, mask, seed=5100 + S + D)[0])


def test_masked_bwd_empty_tiles_are_exact_zeros():
    """Query tile 1 of head 0 keeps nothing (its dQ rows are 0); key tile 3 is
    dropped for every query tile (its dK, dV rows are 0)."""
    S, Hq = 600, 2
    nt = (S + 127) // 128
    mask = np.ones((Hq, nt, nt), np.uint8)
    mask[0, 1, :] = 0
    mask[:, :, 3] = 0
    _, (dq, dk, dv, rq, rk, rv) = _check(1, Hq, Hq, S, 128, True, mask, seed=5200)
    assert np.all(dq[0, 0, 128:256] == 0) and np.all(rq[0, 0, 128:256] == 0)
    assert np.all(dk[0, :, 384:512] == 0) and np.all(dv[0, :, 384:512] == 0)


def test_masked_bwd_all_ones_equals_unmasked():
    B, Hq, Hkv, S, D = 2, 4, 2, 700, 128
    q, k, v = qkv_bf16(B, Hq, Hkv, S, D, seed=5300)
    do = gaussian_bf16((B, Hq, S, D), 5300, 3)
    nt = (S + 127) // 128
    a = run_gpu_bwd_masked(q, k, v, do, 0.088, True, np.ones((1, nt, nt), np.uint8))
    b = run_gpu_bwd(q, k, v, do, 0.088, True)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("w", WORKLOADS[1:], ids=lambda w: w.name)
def test_masked_bwd_full_size_sampled_heads(w):
    mask = random_block_mask(w.Hq, w.S, 0.5, seed=w.seed)
    heads = [0, w.B * w.Hkv - 1]
    print(w.name, _check(w.B, w.Hq, w.Hkv, w.S, w.D, True, mask, seed=w.seed, kv_heads=heads,
                         sigma=w.sigma)[0])


@pytest.mark.parametrize("density", [0.0, 0.1])
def test_masked_bwd_sparse_masks_many_empty_units(density):
    """Most (or all) units of both kernels keep nothing: consecutive empty units
    must stay in step with the element-wise warps.  All-zero mask: every
    gradient is exactly 0."""
    B, Hq, Hkv, S, D = 1, 32, 32, 2048, 128
    mask = random_block_mask(Hq, S, density, seed=5400)
    q, k, v = qkv_bf16(B, Hq, Hkv, S, D, seed=5400)
    do = gaussian_bf16((B, Hq, S, D), 5400, 3)
    _, _, dq, dk, dv, _ = run_gpu_bwd_masked(q, k, v, do, D ** -0.5, True, mask)
    if density == 0.0:
        assert not dq.any() and not dk.any() and not dv.any()
        return
    heads = [0, 13, 31]
    rq, rk, rv, _ = oracle.attention_bwd(q, k, v, do, D ** -0.5, True, kv_heads=heads, block_mask=mask)
    sel = np.asarray(heads)
    compare_grad(dq.reshape(B * Hkv, 1, S, D)[sel], rq, "sparse dQ")
    compare_grad(dk.reshape(B * Hkv, S, D)[sel], rk, "sparse dK")
    compare_grad(dv.reshape(B * Hkv, S, D)[sel], rv, "sparse dV")
