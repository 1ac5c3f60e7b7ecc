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


def _direct_ex(q, k, v, do, scale, kb, p):
    """(O, LSE, dQ, dK, dV) from attn_fwd_ex / attn_bwd_ex called directly."""
    import torch
    from causal_scaled_dot_gb300 import native
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    qd, kd, vd, dod = (to_device(x) for x in (q, k, v, do))
    kbd = torch.from_numpy(kb).cuda()
    opts = native.options(keep_bits=kbd, dropout_p=p, seed=5, offset=6)
    out = torch.empty_like(qd)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    native.attn_fwd_ex(qd, kd, vd, out, lse, B, Hq, Hkv, S, D, scale, True, opts)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    delta = torch.empty_like(lse)
    native.attn_bwd_ex(qd, kd, vd, out, dod, lse, delta, dq, dk, dv, B, Hq, Hkv, S, D, scale, True, opts)
    torch.cuda.synchronize()
    return tuple(t.double().cpu().numpy() for t in (out, lse, dq, dk, dv))


@pytest.mark.parametrize("variant", ["plain", "block", "keep", "dropout", "keep+dropout"])
def test_autograd_matches_direct_backward(variant):
    import torch
    from causal_scaled_dot_gb300 import native
    B, Hq, Hkv, S, D = 2, 4, 2, 300, 128
    q, k, v = qkv_bf16(B, Hq, Hkv, S, D, seed=9100)
    do = gaussian_bf16((B, Hq, S, D), 9100, 3)
    scale = 1.0 / math.sqrt(D)
    bm = random_block_mask(Hq, S, 0.7, seed=91) if variant == "block" else None
    kb = random_keep_bits(1, S, 0.6, seed=92) if "keep" in variant else None
    p = 0.2 if "dropout" in variant else 0.0
    tq, tk, tv = (to_device(x).requires_grad_() for x in (q, k, v))
    o = native.attention_trainable(tq, tk, tv, True, scale,
                                   block_mask=None if bm is None else torch.from_numpy(bm).cuda(),
                                   keep_bits=None if kb is None else torch.from_numpy(kb).cuda(),
                                   dropout_p=p, seed=5, offset=6, check_status=True)
    o.backward(to_device(do))
    got = [t.grad.double().cpu().numpy() for t in (tq, tk, tv)]
    if variant == "plain":
        want = run_gpu_bwd(q, k, v, do, scale, True)
    elif variant == "block":
        want = run_gpu_bwd_masked(q, k, v, do, scale, True, bm)
    elif variant == "keep":
        want = run_gpu_bwd_elem_masked(q, k, v, do, scale, True, kb)
    elif variant == "keep+dropout":
        want = _direct_ex(q, k, v, do, scale, kb, p)
    else:
        want = run_gpu_bwd_dropout(q, k, v, do, scale, True, p, 5, 6)
    assert np.array_equal(o.detach().double().cpu().numpy(), want[0])
    for g, w_ in zip(got, want[2:5]):
        assert np.array_equal(g, w_)


def test_entry_points_from_a_thread_with_no_cuda_call():
    """A thread that has made no CUDA call has no driver context bound (the
    autograd engine's worker is one); the forward and backward entry points
    called from such a thread give the same bits as from the main thread."""
    import threading

    import torch
    from causal_scaled_dot_gb300 import native
    B, Hq, Hkv, S, D = 1, 2, 1, 200, 64
    q, k, v = (to_device(x) for x in qkv_bf16(B, Hq, Hkv, S, D, seed=9200))
    do = to_device(gaussian_bf16((B, Hq, S, D), 9200, 3))
    scale = 1.0 / math.sqrt(D)

    def buffers():
        lse = torch.empty((B, Hq, S), device=q.device, dtype=torch.float32)
        return (torch.empty_like(q), lse, torch.empty_like(lse), torch.empty_like(q),
                torch.empty_like(k), torch.empty_like(v))

    def run(bufs, stream):
        o, lse, delta, dq, dk, dv = bufs
        native.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, S, D, scale, True, stream=stream)
        native.attn_bwd(q, k, v, o, do, lse, delta, dq, dk, dv, B, Hq, Hkv, S, D, scale, True,
                        stream=stream)

    side = torch.cuda.Stream()
    handle = side.cuda_stream  # an int: the thread itself touches no torch CUDA state
    in_thread, in_main = buffers(), buffers()
    torch.cuda.synchronize()
    errors = []

    def worker():
        try:
            run(in_thread, handle)
        except Exception as e:  # re-raised in the main thread below
            errors.append(e)

    t = threading.Thread(target=worker)
    t.start()
    t.join()
    side.synchronize()
    assert not errors, errors
    run(in_main, handle)
    side.synchronize()
    for a, b in zip(in_thread, in_main):
        assert torch.equal(a, b)


def test_attention_wrapper_with_status_check():
    """``attention`` runs on the tensors' device with its current stream and,
    with check_status, reads the status word: the result equals the direct call."""
    import torch
    from causal_scaled_dot_gb300 import native
    B, Hq, Hkv, S, D = 1, 2, 2, 257, 128
    q, k, v = (to_device(x) for x in qkv_bf16(B, Hq, Hkv, S, D, seed=9300))
    o, lse = native.attention(q, k, v, True, check_status=True)
    o2, lse2 = torch.empty_like(q), torch.empty_like(lse)
    native.attn_fwd(q, k, v, o2, lse2, B, Hq, Hkv, S, D, 1.0 / math.sqrt(D), True)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
