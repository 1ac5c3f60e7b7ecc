"""GPU parity of the FP8 (E4M3) entry point against the fp64 oracle on the same
codes and descales.  Tolerances: the worst-case bounds of
tests/gpu_util.fp8_tolerances, with the relative L2 bound tightened to twice
the error that rounding the exact weights to E4M3 gives on the same inputs
(tests/gpu_util.fp8_rounding_model) plus the output rounding."""
import math

import numpy as np
import pytest

import oracle
from causal_scaled_dot_gb300.inputs import qkv_e4m3
from causal_scaled_dot_gb300.workloads import WORKLOADS
from tests.gpu_util import compare_fp8, fp8_rounding_model, run_gpu_fp8, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _check(B, Hq, Hkv, S, causal, seed, descales=(1.0, 1.0, 1.0), sigma=1.0, rows=None):
    D = 128
    q, k, v = qkv_e4m3(B, Hq, Hkv, S, D, seed=seed, sigma=sigma)
    descales = tuple(float(np.float32(d)) for d in descales)
    scale = 1.0 / math.sqrt(D)
    o, l = run_gpu_fp8(q, k, v, descales, scale, causal)
    o_ref, l_ref = oracle.attention_e4m3(q, k, v, scale, descales, causal, rows=rows)
    vals = oracle.e4m3_decode(v) * descales[2]
    model = fp8_rounding_model(q, k, v, descales, scale, causal, rows)
    if rows is not None:
        o, l = o.reshape(-1, D)[rows], l.reshape(-1)[rows]
    return compare_fp8(o, o_ref, l, l_ref, vals, f"fp8 B{B} Hq{Hq} Hkv{Hkv} S{S} causal={causal}",
                       model_rel=model)


@pytest.mark.parametrize("S", [1, 2, 127, 128, 129, 300, 1000])
@pytest.mark.parametrize("causal", [True, False])
def test_fp8_sequence_lengths(S, causal):
    _check(1, 2, 1, S, causal, seed=1100 + S)


@pytest.mark.parametrize("Hq,Hkv,B", [(4, 4, 1), (8, 2, 3), (32, 1, 1)])
def test_fp8_heads_and_batches(Hq, Hkv, B):
    _check(B, Hq, Hkv, 250, True, seed=1200 + Hq + Hkv + B)


def test_fp8_descales():
    """Non-unit descales: the Q and K descales act through the softmax scale, the
    V descale on the output."""
    _check(2, 4, 2, 400, True, seed=1301, descales=(0.37, 2.5, 0.61))


@pytest.mark.parametrize("w", WORKLOADS[1:], ids=lambda w: w.name)
def test_fp8_full_size_workloads_sampled_rows(w):
    rows = sample_rows(w.B, w.Hq, w.S, n_random=256, seed=w.seed)
    print(w.name, _check(w.B, w.Hq, w.Hkv, w.S, True, seed=w.seed, sigma=w.sigma, rows=rows))


def test_fp8_causal_row0_equals_v0():
    """Row 0 attends to key 0 only (weight exactly 1 in E4M3): O_0 = descale * V_0."""
    q, k, v = qkv_e4m3(1, 2, 2, 200, 128, seed=1401)
    o, _ = run_gpu_fp8(q, k, v, (1.0, 1.0, 0.5), 1 / math.sqrt(128), True)
    v0 = oracle.e4m3_decode(v[:, :, 0, :]) * 0.5
    assert np.array_equal(o[:, :, 0, :], v0)
