"""The autograd wrapper over the C ABI (native.attention_trainable): its
gradients are exactly those of the direct backward calls, for every variant."""
import math

import numpy as np
import pytest

from causal_scaled_dot_gb300.inputs import (gaussian_bf16, qkv_bf16, random_block_mask,
                                            random_keep_bits)
from tests.gpu_util import (run_gpu_bwd, run_gpu_bwd_dropout, run_gpu_bwd_elem_masked,
                            run_gpu_bwd_masked, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("variant", ["plain", "block", "keep", "dropout"])
def test_autograd_matches_direct_backward(variant):
    import torch
    from causal_scaled_dot_gb300 import native
    B, Hq, Hkv, S, D = 2, 4, 2, 300, 128
    q, k, v = qkv_bf16(B, Hq, Hkv, S, D, seed=9100)
    do = gaussian_bf16((B, Hq, S, D), 9100, 3)
    scale = 1.0 / math.sqrt(D)
    bm = random_block_mask(Hq, S, 0.7, seed=91) if variant == "block" else None
    kb = random_keep_bits(1, S, 0.6, seed=92) if variant == "keep" else None
    p = 0.2 if variant == "dropout" else 0.0
    tq, tk, tv = (to_device(x).requires_grad_() for x in (q, k, v))
    o = native.attention_trainable(tq, tk, tv, True, scale,
                                   block_mask=None if bm is None else torch.from_numpy(bm).cuda(),
                                   keep_bits=None if kb is None else torch.from_numpy(kb).cuda(),
                                   dropout_p=p, seed=5, offset=6)
    o.backward(to_device(do))
    got = [t.grad.double().cpu().numpy() for t in (tq, tk, tv)]
    if variant == "plain":
        want = run_gpu_bwd(q, k, v, do, scale, True)
    elif variant == "block":
        want = run_gpu_bwd_masked(q, k, v, do, scale, True, bm)
    elif variant == "keep":
        want = run_gpu_bwd_elem_masked(q, k, v, do, scale, True, kb)
    else:
        want = run_gpu_bwd_dropout(q, k, v, do, scale, True, p, 5, 6)
    assert np.array_equal(o.detach().double().cpu().numpy(), want[0])
    for g, w_ in zip(got, want[2:5]):
        assert np.array_equal(g, w_)
