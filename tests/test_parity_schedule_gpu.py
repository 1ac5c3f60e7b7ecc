"""GPU parity on both work orders of the persistent forward kernel: the host's
table (attn_fwd_schedule; every shape up to 4096 units) and the arithmetic
boustrophedon order the kernel falls back to beyond it.  Heads are
independent, so the many-head shapes are checked against the fp64 oracle on
slices of heads (first, middle and last ones)."""
import math

import numpy as np
import pytest

import oracle
from causal_scaled_dot_gb300 import native
from causal_scaled_dot_gb300.inputs import qkv_bf16
from tests.gpu_util import compare, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _check_heads(q, k, v, o, l, scale, causal, heads, label):
    group = q.shape[1] // k.shape[1]
    for h in heads:
        kh = h // group
        o_ref, l_ref = oracle.attention(q[:, h:h + 1], k[:, kh:kh + 1], v[:, kh:kh + 1], scale, causal)
        compare(o[:, h:h + 1], o_ref, l[:, h:h + 1], l_ref, f"{label} head {h}")


@pytest.mark.parametrize("Hq,Hkv,S,D,causal,table", [
    (2100, 2100, 300, 64, True, False),   # 2100 x 2 = 4200 units: arithmetic order
    (2080, 520, 300, 64, True, False),    # 2080 x 2 = 4160 units, GQA 4:1
    (2048, 2048, 300, 64, True, True),    # 2048 x 2 = 4096 units: the largest table
    (48, 48, 1900, 128, True, True),      # 384 units, 15 query tiles (a ragged pair)
    (48, 48, 1000, 128, False, False),    # non-causal, 192 units: under two per CTA
    (80, 80, 1000, 128, False, True),     # non-causal, 320 units
])
def test_work_orders(Hq, Hkv, S, D, causal, table):
    nq = (S + 127) // 128
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    units = Hq * ((nq + 1) // 2)
    assert (native.fwd_schedule(Hq, nq, causal, min(units, sms)) is not None) == table
    q, k, v = qkv_bf16(1, Hq, Hkv, S, D, seed=8100 + Hq)
    scale = 1.0 / math.sqrt(D)
    o, l, _ = run_gpu(q, k, v, scale, causal)
    heads = sorted({0, 1, Hq // 2, Hq - 2, Hq - 1})
    _check_heads(q, k, v, o, l, scale, causal, heads, f"Hq{Hq} S{S} table={table}")
