"""GPU parity of the backward entry point (attn_bwd, after attn_fwd on the same
inputs) against the fp64 oracle's gradients.  Tolerances: tests/gpu_util
(relative L2 <= 1e-2 and max error <= 2 % of the largest magnitude per tensor;
delta within one bf16 rounding of O per row)."""
import math

import numpy as np
import pytest

import oracle
from causal_scaled_dot_gb300.inputs import bf16_bits_to_float32, gaussian_bf16, qkv_bf16
from causal_scaled_dot_gb300.workloads import WORKLOADS
from tests.gpu_util import compare_delta, compare_grad, run_gpu_bwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _inputs(B, Hq, Hkv, S, D, seed, sigma=1.0):
    q, k, v = qkv_bf16(B, Hq, Hkv, S, D, seed=seed, sigma=sigma)
    do = gaussian_bf16((B, Hq, S, D), seed, 3)
    return q, k, v, do


def _check(B, Hq, Hkv, S, D, causal, seed, sigma=1.0, kv_heads=None):
    q, k, v, do = _inputs(B, Hq, Hkv, S, D, seed, sigma)
    scale = 1.0 / math.sqrt(D)
    O, L, dq, dk, dv, delta = run_gpu_bwd(q, k, v, do, scale, causal)
    rq, rk, rv, rdelta = oracle.attention_bwd(q, k, v, do, scale, causal, kv_heads=kv_heads)
    o_ref, _ = oracle.attention(q, k, v, scale, causal)
    G = Hq // Hkv
    do64 = bf16_bits_to_float32(do).astype(np.float64)
    if kv_heads is not None:
        sel = np.asarray(kv_heads)
        dq = dq.reshape(B * Hkv, G, S, D)[sel]
        delta = delta.reshape(B * Hkv, G, S)[sel]
        dk = dk.reshape(B * Hkv, S, D)[sel]
        dv = dv.reshape(B * Hkv, S, D)[sel]
        o_ref = o_ref.reshape(B * Hkv, G, S, D)[sel]
        do64 = do64.reshape(B * Hkv, G, S, D)[sel]
    label = f"bwd B{B} Hq{Hq} Hkv{Hkv} S{S} D{D} causal={causal}"
    return {"dq": compare_grad(dq, rq, label + " dQ"), "dk": compare_grad(dk, rk, label + " dK"),
            "dv": compare_grad(dv, rv, label + " dV"),
            "delta": compare_delta(delta, rdelta, o_ref, do64, label + " delta")}


@pytest.mark.parametrize("S", [1, 2, 127, 128, 129, 300, 1000])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_bwd_sequence_lengths(S, D, causal):
    print(_check(1, 2, 1, S, D, causal, seed=2100 + S + D))


@pytest.mark.parametrize("Hq,Hkv,B", [(4, 4, 1), (8, 2, 3), (32, 1, 1), (4, 2, 2)])
def test_bwd_heads_and_batches(Hq, Hkv, B):
    print(_check(B, Hq, Hkv, 250, 128, True, seed=2200 + Hq + Hkv + B))


def test_bwd_many_units():
    """More units than SMs in both kernels, several rounds each."""
    print(_check(2, 8, 4, 2048, 128, True, seed=2300, kv_heads=[0, 7]))


@pytest.mark.parametrize("w", WORKLOADS[1:], ids=lambda w: w.name)
def test_bwd_full_size_workloads_sampled_heads(w):
    """The full-size backward on the GPU; the oracle's gradients of the first
    and last key/value heads (every query head of their groups)."""
    heads = [0, w.B * w.Hkv - 1]
    print(w.name, _check(w.B, w.Hq, w.Hkv, w.S, w.D, True, seed=w.seed, sigma=w.sigma,
                         kv_heads=heads))


def test_bwd_repeated_calls_are_bitwise_equal():
    q, k, v, do = _inputs(1, 4, 2, 700, 128, 2400)
    a = run_gpu_bwd(q, k, v, do, 0.088, True)
    b = run_gpu_bwd(q, k, v, do, 0.088, True)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
