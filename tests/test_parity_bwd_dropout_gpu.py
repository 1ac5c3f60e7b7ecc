"""GPU parity of the backward with dropout (attn_bwd_dropout after
attn_fwd_dropout) against the oracle's gradients with the same keep decisions,
with the tolerances of the unmasked backward (tests/gpu_util)."""
import math

import numpy as np
import pytest

import oracle
from causal_scaled_dot_gb300.inputs import gaussian_bf16, qkv_bf16
from causal_scaled_dot_gb300.workloads import WORKLOADS
from causal_scaled_dot_gb300.inputs import bf16_bits_to_float32
from tests.gpu_util import compare_grad, run_gpu_bwd, run_gpu_bwd_dropout

pytestmark = pytest.mark.gpu

SEED, OFFSET = 0x5EED5EED1234, 77


def f64(bits):
    return bf16_bits_to_float32(bits).astype(np.float64)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _check(B, Hq, Hkv, S, D, causal, p, seed, kv_heads=None, sigma=1.0):
    q, k, v = qkv_bf16(B, Hq, Hkv, S, D, seed=seed, sigma=sigma)
    do = gaussian_bf16((B, Hq, S, D), seed, 3)
    scale = 1.0 / math.sqrt(D)
    p8 = int(round(p * 256))
    o, _, dq, dk, dv, _ = run_gpu_bwd_dropout(q, k, v, do, scale, causal, p, SEED, OFFSET)
    rq, rk, rv, _ = oracle.attention_bwd(q, k, v, do, scale, causal, kv_heads=kv_heads,
                                         dropout=(p8, SEED, OFFSET))
    G = Hq // Hkv
    # delta = dO . O is formed from the bf16 output O, which here holds the kept
    # values scaled by 256/(256-p8) and so is rounded (without dropout O is an
    # exact bf16 average for a single key).  Its error e_i <= 2^-8 sum_d |dO O|
    # reaches dQ_i as scale * e_i * (P K)_i and dK_j as scale * sum_i P_ij e_i Q_i:
    # an additive error that matters where the exact gradient is 0 (a single
    # key); for dK the bound takes one unit of weight per query head.
    e = 2.0 ** -8 * float(np.max(np.sum(np.abs(f64(do) * o), axis=-1)))
    err_q = scale * e * float(np.max(np.abs(f64(k))))
    err_k = scale * e * float(np.max(np.abs(f64(q)))) * G
    if kv_heads is not None:
        sel = np.asarray(kv_heads)
        dq = dq.reshape(B * Hkv, G, S, D)[sel]
        dk = dk.reshape(B * Hkv, S, D)[sel]
        dv = dv.reshape(B * Hkv, S, D)[sel]
    label = f"dropout bwd p={p} B{B} Hq{Hq} Hkv{Hkv} S{S} D{D} causal={causal}"
    return {"dq": compare_grad(dq, rq, label + " dQ", err_q), "dk": compare_grad(dk, rk, label + " dK", err_k),
            "dv": compare_grad(dv, rv, label + " dV")}, (dq, dk, dv)


@pytest.mark.parametrize("S", [1, 129, 300, 1000])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("p", [0.1, 0.5])
def test_dropout_bwd(S, D, causal, p):
    print(_check(2, 4, 2, S, D, causal, p, seed=8100 + S + D)[0])


def test_dropout_bwd_high_rate():
    print(_check(1, 2, 2, 700, 128, True, 0.9, seed=8200)[0])


def test_dropout_bwd_zero_rate_equals_plain_backward():
    B, Hq, Hkv, S, D = 2, 4, 2, 300, 128
    q, k, v = qkv_bf16(B, Hq, Hkv, S, D, seed=8300)
    do = gaussian_bf16((B, Hq, S, D), 8300, 3)
    a = run_gpu_bwd_dropout(q, k, v, do, 0.088, True, 0.0, SEED, OFFSET)
    b = run_gpu_bwd(q, k, v, do, 0.088, True)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_dropout_bwd_deterministic_and_seeded():
    B, Hq, Hkv, S, D = 1, 2, 2, 400, 64
    q, k, v = qkv_bf16(B, Hq, Hkv, S, D, seed=8400)
    do = gaussian_bf16((B, Hq, S, D), 8400, 3)
    a = run_gpu_bwd_dropout(q, k, v, do, 0.125, True, 0.2, SEED, OFFSET)
    b = run_gpu_bwd_dropout(q, k, v, do, 0.125, True, 0.2, SEED, OFFSET)
    c = run_gpu_bwd_dropout(q, k, v, do, 0.125, True, 0.2, SEED + 1, OFFSET)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    assert not np.array_equal(a[4], c[4])


@pytest.mark.parametrize("w", WORKLOADS[1:], ids=lambda w: w.name)
def test_dropout_bwd_full_size_sampled_heads(w):
    """The launch the benchmark times (p = 0.1) on the first and last key/value heads."""
    heads = [0, w.B * w.Hkv - 1]
    print(w.name, _check(w.B, w.Hq, w.Hkv, w.S, w.D, True, 0.1, seed=w.seed, kv_heads=heads,
                         sigma=w.sigma)[0])
