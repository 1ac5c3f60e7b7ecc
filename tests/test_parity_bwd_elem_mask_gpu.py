"""GPU parity of the element-masked backward (attn_bwd_elem_masked after
attn_fwd_elem_masked) against the oracle's element-masked gradients, with the
tolerances of the unmasked backward (tests/gpu_util).  Includes rows that see
no key (their dQ is exactly 0) and the all-ones mask against attn_bwd."""
import math

import numpy as np
import pytest

import oracle
from causal_scaled_dot_gb300.inputs import (block_mask_of_keep_bits, gaussian_bf16, pack_keep_bits,
                                            qkv_bf16, random_block_mask, random_keep_bits,
                                            window_keep_bits)
from causal_scaled_dot_gb300.workloads import WORKLOADS
from tests.gpu_util import compare_grad, run_gpu_bwd, run_gpu_bwd_elem_masked

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _check(B, Hq, Hkv, S, D, causal, bits, seed, block_mask=None, kv_heads=None, sigma=1.0):
    q, k, v = qkv_bf16(B, Hq, Hkv, S, D, seed=seed, sigma=sigma)
    do = gaussian_bf16((B, Hq, S, D), seed, 3)
    scale = 1.0 / math.sqrt(D)
    _, _, dq, dk, dv, _ = run_gpu_bwd_elem_masked(q, k, v, do, scale, causal, bits, block_mask)
    rq, rk, rv, _ = oracle.attention_bwd(q, k, v, do, scale, causal, kv_heads=kv_heads,
                                         block_mask=block_mask, keep_bits=bits)
    G = Hq // Hkv
    if kv_heads is not None:
        sel = np.asarray(kv_heads)
        dq = dq.reshape(B * Hkv, G, S, D)[sel]
        dk = dk.reshape(B * Hkv, S, D)[sel]
        dv = dv.reshape(B * Hkv, S, D)[sel]
    label = f"elem-masked bwd B{B} Hq{Hq} Hkv{Hkv} S{S} D{D} causal={causal} Hm={bits.shape[0]}"
    return {"dq": compare_grad(dq, rq, label + " dQ"), "dk": compare_grad(dk, rk, label + " dK"),
            "dv": compare_grad(dv, rv, label + " dV")}, (dq, dk, dv, rq, rk, rv)


@pytest.mark.parametrize("S", [129, 300, 1000])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("density", [0.2, 0.7])
def test_elem_masked_bwd_random(S, D, causal, density):
    Hq = 4
    per_head = (S + D) % 2 == 0
    bits = random_keep_bits(Hq if per_head else 1, S, density, seed=S + D + int(100 * density) + 1)
    print(_check(2, Hq, 2, S, D, causal, bits, seed=7100 + S + D)[0])


def test_elem_masked_bwd_rows_without_keys():
    S, Hq = 300, 2
    rng = np.random.default_rng(7)
    keep = rng.random((Hq, S, S)) < 0.4
    keep[:, np.arange(S), np.arange(S)] = True
    keep[1, 3, :] = False
    keep[0, 32:64, :] = False
    _, (dq, dk, dv, rq, rk, rv) = _check(1, Hq, Hq, S, 128, True, pack_keep_bits(keep), seed=7200)
    assert np.all(dq[0, 1, 3] == 0) and np.all(dq[0, 0, 32:64] == 0)


@pytest.mark.parametrize("window", [1, 200, 700])
def test_elem_masked_bwd_window(window):
    S = 1000
    bits = window_keep_bits(S, window)
    bm = block_mask_of_keep_bits(bits, S)
    print(_check(1, 4, 2, S, 128, True, bits, seed=7300 + window, block_mask=bm)[0])
    print(_check(1, 4, 2, S, 64, True, bits, seed=7310 + window)[0])


def test_elem_masked_bwd_with_random_block_mask():
    S, Hq = 700, 4
    bits = random_keep_bits(Hq, S, 0.6, seed=74)
    bm = random_block_mask(Hq, S, 0.6, seed=75)
    print(_check(2, Hq, 2, S, 128, True, bits, seed=7400, block_mask=bm)[0])


def test_elem_masked_bwd_all_ones_equals_unmasked():
    B, Hq, Hkv, S, D = 2, 4, 2, 700, 128
    q, k, v = qkv_bf16(B, Hq, Hkv, S, D, seed=7500)
    do = gaussian_bf16((B, Hq, S, D), 7500, 3)
    ones = np.full((1, S, 16 * ((S + 127) // 128)), 0xFF, np.uint8)
    a = run_gpu_bwd_elem_masked(q, k, v, do, 0.088, True, ones)
    b = run_gpu_bwd(q, k, v, do, 0.088, True)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("w", WORKLOADS[1:], ids=lambda w: w.name)
def test_elem_masked_bwd_full_size_sampled_heads(w):
    """The launch the benchmark times: a 1024-key local window with its block mask."""
    bits = window_keep_bits(w.S, 1024)
    bm = block_mask_of_keep_bits(bits, w.S)
    heads = [0, w.B * w.Hkv - 1]
    print(w.name, _check(w.B, w.Hq, w.Hkv, w.S, w.D, True, bits, seed=w.seed, block_mask=bm,
                         kv_heads=heads, sigma=w.sigma)[0])
