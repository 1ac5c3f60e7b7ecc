"""GPU parity of the combined options (attn_fwd_ex / attn_bwd_ex) against the
oracle's combined variants: masks with dropout, masks with E4M3 inputs, and the
gradients of block masks and keep bits with dropout; single options through the
options entry equal their own entry points bit for bit."""
import math

import numpy as np
import pytest

import oracle
from causal_scaled_dot_gb300.inputs import (bf16_bits_to_float32, gaussian_bf16, qkv_bf16, qkv_e4m3,
                                            random_block_mask, random_keep_bits)
from causal_scaled_dot_gb300.workloads import WORKLOADS
from tests.gpu_util import (compare_fp8, compare_grad, compare_masked, run_gpu_bwd_dropout,
                            run_gpu_dropout, run_gpu_elem_masked, to_device)

pytestmark = pytest.mark.gpu

SEED, OFFSET = 0xC0FFEE, 11


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _dev(x):
    import torch
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).cuda()


def run_fwd_ex(q, k, v, scale, causal, descales=None, bm=None, kb=None, p=0.0):
    import torch
    from causal_scaled_dot_gb300 import native
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    dev = _dev if descales is not None else to_device
    qd, kd, vd = dev(q), dev(k), dev(v)
    out = torch.full((B, Hq, S, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device="cuda")
    bmd, kbd = _dev(bm), _dev(kb)
    opts = native.options(e4m3_descales=descales, block_mask=bmd, keep_bits=kbd, dropout_p=p, seed=SEED,
                          offset=OFFSET)
    native.attn_fwd_ex(qd, kd, vd, out, lse, B, Hq, Hkv, S, D, scale, causal, opts)
    native.attn_sync_status(None)
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


@pytest.mark.parametrize("S", [129, 700])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("combo", ["block+dropout", "keep+dropout", "block+keep+dropout"])
def test_fwd_masks_with_dropout(S, D, causal, combo):
    Hq, Hkv, p = 4, 2, 0.2
    q, k, v = qkv_bf16(2, Hq, Hkv, S, D, seed=9300 + S + D)
    bm = random_block_mask(Hq, S, 0.7, seed=S) if "block" in combo else None
    kb = random_keep_bits(1, S, 0.7, seed=S + 1) if "keep" in combo else None
    scale = 1 / math.sqrt(D)
    o, l = run_fwd_ex(q, k, v, scale, causal, bm=bm, kb=kb, p=p)
    ro, rl = oracle.attention_ex(q, k, v, scale, causal, block_mask=bm, keep_bits=kb,
                                 dropout=(int(round(p * 256)), SEED, OFFSET))
    p8 = int(round(p * 256))
    print(compare_masked(o, ro, l, rl, f"{combo} S{S} D{D} causal={causal}", abs_scale=256 / (256 - p8)))


@pytest.mark.parametrize("combo", ["block", "keep", "block+keep"])
@pytest.mark.parametrize("causal", [True, False])
def test_fwd_e4m3_with_masks(combo, causal):
    Hq, Hkv, S, D = 4, 2, 700, 128
    q, k, v = qkv_e4m3(2, Hq, Hkv, S, D, seed=9400)
    ds = (0.5, 1.5, 0.75)
    bm = random_block_mask(Hq, S, 0.6, seed=94) if "block" in combo else None
    kb = random_keep_bits(Hq, S, 0.6, seed=95) if "keep" in combo else None
    o, l = run_fwd_ex(q, k, v, 0.09, causal, descales=ds, bm=bm, kb=kb)
    ro, rl = oracle.attention_ex(q, k, v, 0.09, causal, descales=ds, block_mask=bm, keep_bits=kb)
    vals = oracle.e4m3_decode(v) * ds[2]
    live = ~np.isneginf(rl)
    assert np.all(np.isneginf(l[~live])) and np.all(o[~live] == 0.0)
    print(compare_fp8(o[live], ro[live], l[live], rl[live], vals, f"e4m3 {combo} causal={causal}"))


def test_options_with_one_feature_equal_their_own_entry_points():
    B, Hq, Hkv, S, D = 2, 4, 2, 300, 128
    q, k, v = qkv_bf16(B, Hq, Hkv, S, D, seed=9500)
    kb = random_keep_bits(Hq, S, 0.5, seed=95)
    a = run_fwd_ex(q, k, v, 0.088, True, kb=kb)
    b = run_gpu_elem_masked(q, k, v, 0.088, True, kb)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    a = run_fwd_ex(q, k, v, 0.088, True, p=0.3)
    b = run_gpu_dropout(q, k, v, 0.088, True, 0.3, SEED, OFFSET)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def _bwd_ex(q, k, v, do, scale, causal, bm, p, kb=None):
    import torch
    from causal_scaled_dot_gb300 import native
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    qd, kd, vd, dod = to_device(q), to_device(k), to_device(v), to_device(do)
    out = torch.empty_like(qd)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    bmd, kbd = _dev(bm), _dev(kb)
    opts = native.options(block_mask=bmd, keep_bits=kbd, dropout_p=p, seed=SEED, offset=OFFSET)
    native.attn_fwd_ex(qd, kd, vd, out, lse, B, Hq, Hkv, S, D, scale, causal, opts)
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in (qd, kd, vd))
    delta = torch.full_like(lse, float("nan"))
    native.attn_bwd_ex(qd, kd, vd, out, dod, lse, delta, dq, dk, dv, B, Hq, Hkv, S, D, scale, causal, opts)
    native.attn_sync_status(None)
    return tuple(t.double().cpu().numpy() for t in (out, lse, dq, dk, dv, delta))


@pytest.mark.parametrize("S", [129, 700])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_bwd_block_mask_with_dropout(S, D, causal):
    Hq, Hkv, p = 4, 2, 0.2
    q, k, v = qkv_bf16(2, Hq, Hkv, S, D, seed=9600 + S + D)
    do = gaussian_bf16((2, Hq, S, D), 9600 + S + D, 3)
    bm = random_block_mask(Hq, S, 0.7, seed=S + 2)
    scale = 1 / math.sqrt(D)
    o, _, dq, dk, dv, _ = _bwd_ex(q, k, v, do, scale, causal, bm, p)
    rq, rk, rv, _ = oracle.attention_bwd(q, k, v, do, scale, causal, block_mask=bm,
                                         dropout=(int(round(p * 256)), SEED, OFFSET))
    # delta from the rounded bf16 output (see tests/test_parity_bwd_dropout_gpu.py)
    f64 = lambda b: bf16_bits_to_float32(b).astype(np.float64)  # noqa: E731
    e = 2.0 ** -8 * float(np.max(np.sum(np.abs(f64(do) * o), axis=-1)))
    label = f"block+dropout bwd S{S} D{D} causal={causal}"
    print(compare_grad(dq, rq, label + " dQ", scale * e * float(np.max(np.abs(f64(k))))),
          compare_grad(dk, rk, label + " dK", scale * e * float(np.max(np.abs(f64(q)))) * 2),
          compare_grad(dv, rv, label + " dV"))


def _check_bwd_combo(q, k, v, do, scale, causal, bm, kb, p, label):
    o, _, dq, dk, dv, _ = _bwd_ex(q, k, v, do, scale, causal, bm, p, kb)
    rq, rk, rv, _ = oracle.attention_bwd(q, k, v, do, scale, causal, block_mask=bm, keep_bits=kb,
                                         dropout=(int(round(p * 256)), SEED, OFFSET))
    # delta from the rounded bf16 output, as in test_bwd_block_mask_with_dropout
    f64 = lambda b: bf16_bits_to_float32(b).astype(np.float64)  # noqa: E731
    e = 2.0 ** -8 * float(np.max(np.sum(np.abs(f64(do) * o), axis=-1)))
    return (compare_grad(dq, rq, label + " dQ", scale * e * float(np.max(np.abs(f64(k))))),
            compare_grad(dk, rk, label + " dK", scale * e * float(np.max(np.abs(f64(q)))) * 2),
            compare_grad(dv, rv, label + " dV"))


@pytest.mark.parametrize("S", [129, 700])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("combo", ["keep+dropout", "block+keep+dropout"])
def test_bwd_keep_bits_with_dropout(S, D, causal, combo):
    Hq, Hkv, p = 4, 2, 0.2
    q, k, v = qkv_bf16(2, Hq, Hkv, S, D, seed=9800 + S + D)
    do = gaussian_bf16((2, Hq, S, D), 9800 + S + D, 3)
    kb = random_keep_bits(1 if D == 64 else Hq, S, 0.7, seed=S + 3)
    bm = random_block_mask(Hq, S, 0.7, seed=S + 4) if "block" in combo else None
    print(_check_bwd_combo(q, k, v, do, 1 / math.sqrt(D), causal, bm, kb, p,
                           f"{combo} bwd S{S} D{D} causal={causal}"))


def test_bwd_keep_bits_with_dropout_on_a_window():
    """A 256-key local window (rows that see few keys) with dropout 0.1, GQA 4:1."""
    from causal_scaled_dot_gb300.inputs import block_mask_of_keep_bits, window_keep_bits
    B, Hq, Hkv, S, D = 1, 8, 2, 1000, 128
    q, k, v = qkv_bf16(B, Hq, Hkv, S, D, seed=9900)
    do = gaussian_bf16((B, Hq, S, D), 9900, 3)
    kb = window_keep_bits(S, 256)
    bm = block_mask_of_keep_bits(kb, S)
    print(_check_bwd_combo(q, k, v, do, 1 / math.sqrt(D), True, bm, kb, 0.1, "window256+dropout bwd"))


def test_bwd_options_dropout_equals_its_own_entry_point():
    B, Hq, Hkv, S, D = 2, 4, 2, 300, 128
    q, k, v = qkv_bf16(B, Hq, Hkv, S, D, seed=9700)
    do = gaussian_bf16((B, Hq, S, D), 9700, 3)
    a = _bwd_ex(q, k, v, do, 0.088, True, None, 0.25)
    b = run_gpu_bwd_dropout(q, k, v, do, 0.088, True, 0.25, SEED, OFFSET)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("w", [x for x in WORKLOADS[1:] if x.name.startswith(("profile", "gqa"))],
                         ids=lambda w: w.name)
def test_window_with_dropout_full_size(w):
    """A 1024-key local window (keep bits and their block mask) with dropout 0.1
    at a timed size: the forward on sampled rows, the gradients on the first
    and last key/value heads."""
    from causal_scaled_dot_gb300.inputs import block_mask_of_keep_bits, window_keep_bits
    from tests.gpu_util import sample_rows
    p = 0.1
    p8 = int(round(p * 256))
    q, k, v = qkv_bf16(w.B, w.Hq, w.Hkv, w.S, w.D, seed=w.seed, sigma=w.sigma)
    do = gaussian_bf16((w.B, w.Hq, w.S, w.D), w.seed, 3)
    kb = window_keep_bits(w.S, 1024)
    bm = block_mask_of_keep_bits(kb, w.S)
    scale = 1 / math.sqrt(w.D)
    o, l, dq, dk, dv, _ = _bwd_ex(q, k, v, do, scale, True, bm, p, kb)
    rows = sample_rows(w.B, w.Hq, w.S, n_random=128, seed=w.seed)
    ro, rl = oracle.attention_ex(q, k, v, scale, True, block_mask=bm, keep_bits=kb,
                                 dropout=(p8, SEED, OFFSET), rows=rows)
    fwd = compare_masked(o.reshape(-1, w.D)[rows], ro, l.reshape(-1)[rows], rl, f"{w.name} window+dropout",
                         abs_scale=256 / (256 - p8))
    heads = [0, w.B * w.Hkv - 1]
    G = w.Hq // w.Hkv
    rq, rk, rv, _ = oracle.attention_bwd(q, k, v, do, scale, True, kv_heads=heads, block_mask=bm, keep_bits=kb,
                                         dropout=(p8, SEED, OFFSET))
    f64 = lambda b: bf16_bits_to_float32(b).astype(np.float64)  # noqa: E731
    e = 2.0 ** -8 * float(np.max(np.sum(np.abs(f64(do) * o), axis=-1)))
    sel = np.asarray(heads)
    label = f"{w.name} window+dropout bwd"
    print(fwd,
          compare_grad(dq.reshape(w.B * w.Hkv, G, w.S, w.D)[sel], rq, label + " dQ",
                       scale * e * float(np.max(np.abs(f64(k))))),
          compare_grad(dk.reshape(w.B * w.Hkv, w.S, w.D)[sel], rk, label + " dK",
                       scale * e * float(np.max(np.abs(f64(q)))) * G),
          compare_grad(dv.reshape(w.B * w.Hkv, w.S, w.D)[sel], rv, label + " dV"))
