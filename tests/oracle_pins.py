"""Pins for the fp64 oracle: facts fixed by the pages and by mathematics.

Each ``pin_*`` takes ``attn(q_bits, k_bits, v_bits, scale, causal, rows=None)``
returning ``(O, LSE)`` in float64 and raises AssertionError when the callable
disagrees with what the pin fixes.  ``tests/test_oracle_pins.py`` runs them on
the oracle; ``tests/test_oracle_mutants.py`` runs them on copies of the oracle
with planted mistakes and requires that some pin fails for each.

None of these re-types the oracle's own loops: each compares against a
library float64 routine, a closed form, an invariant of the definition, or a
hand-derived worked example (tests/golden/worked_example_s3.json).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

from causal_scaled_dot_gb300.inputs import (bf16_bits_to_float32, float32_to_bf16_bits,
                                            gaussian_bf16)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def bits(x) -> np.ndarray:
    """float values that are exact in bf16 -> bf16 bits (asserts exactness)."""
    x32 = np.asarray(x, dtype=np.float32)
    b = float32_to_bf16_bits(x32)
    assert np.array_equal(bf16_bits_to_float32(b), x32), "value not exact in bf16"
    return b


def f64(b) -> np.ndarray:
    return bf16_bits_to_float32(b).astype(np.float64)


def _rand(shape, seed, stream, sigma=1.0):
    return gaussian_bf16(shape, seed, stream, sigma)


def _grid(shape, rng, lo, hi, step):
    """Random multiples of ``step`` in [lo, hi] (exact in bf16 for small grids)."""
    n = int(round((hi - lo) / step))
    return lo + step * rng.integers(0, n + 1, size=shape)


def _sdpa64(q_b, k_b, v_b, scale, causal):
    """torch's scaled_dot_product_attention on CPU in float64 (a library routine)."""
    q = torch.from_numpy(f64(q_b))
    k = torch.from_numpy(f64(k_b))
    v = torch.from_numpy(f64(v_b))
    G = q.shape[1] // k.shape[1]
    k = k.repeat_interleave(G, dim=1)
    v = v.repeat_interleave(G, dim=1)
    return F.scaled_dot_product_attention(q, k, v, is_causal=causal,
                                          scale=float(np.float32(scale))).numpy()


# ---------------------------------------------------------------------------
def pin_sdpa_library(attn):
    """O equals torch's float64 SDPA (math backend on CPU), causal and not, with GQA."""
    for (B, Hq, Hkv, S, D), causal, seed in [((2, 4, 2, 37, 16), True, 11),
                                             ((1, 3, 3, 29, 8), False, 12),
                                             ((1, 4, 1, 20, 4), True, 13)]:
        q = _rand((B, Hq, S, D), seed, 0)
        k = _rand((B, Hkv, S, D), seed, 1)
        v = _rand((B, Hkv, S, D), seed, 2)
        scale = 1.0 / math.sqrt(D)
        O, _ = attn(q, k, v, scale, causal)
        ref = _sdpa64(q, k, v, scale, causal)
        np.testing.assert_allclose(O, ref, rtol=0, atol=1e-12)


def pin_attention_matrix(attn):
    """With V = identity rows (D >= S) the output row is the attention row itself:
    zero above the diagonal (causal), rows summing to 1, and ratios
    P_ij / P_ik = exp(scale * q_i . (k_j - k_k)) (the softmax closed form)."""
    rng = np.random.default_rng(21)
    S, D = 12, 16
    q = bits(_grid((1, 1, S, D), rng, -1, 1, 0.125))
    k = bits(_grid((1, 1, S, D), rng, -1, 1, 0.125))
    v = np.zeros((1, 1, S, D), np.float32)
    for j in range(S):
        v[0, 0, j, j] = 1.0
    v = bits(v)
    scale = 0.25
    qf, kf = f64(q)[0, 0], f64(k)[0, 0]
    for causal in (True, False):
        O, _ = attn(q, k, v, scale, causal)
        P = O[0, 0, :, :S]
        assert np.all(O[0, 0, :, S:] == 0.0)
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        for i in range(S):
            hi = i + 1 if causal else S
            if causal:
                assert np.all(P[i, hi:] == 0.0), "masked keys must get weight exactly 0"
            assert np.all(P[i, :hi] > 0.0)
            sc = scale * (kf[:hi] @ qf[i])
            expect = np.exp(sc - sc[0])
            np.testing.assert_allclose(P[i, :hi] / P[i, 0], expect, rtol=1e-12, atol=0)


def pin_row0_and_s1(attn):
    """Causal row 0 attends to key 0 only: O_0 = V_0 exactly, LSE_0 = scale q_0.k_0.
    S = 1 (causal or not): O = V, LSE = scale q.k."""
    B, H, S, D = 2, 2, 9, 8
    q, k, v = (_rand((B, H, S, D), 31, t) for t in range(3))
    scale = 0.3
    O, L = attn(q, k, v, scale, True)
    assert np.array_equal(O[:, :, 0, :], f64(v)[:, :, 0, :])
    dots = np.einsum("bhd,bhd->bh", f64(q)[:, :, 0], f64(k)[:, :, 0])
    np.testing.assert_allclose(L[:, :, 0], float(np.float32(scale)) * dots, rtol=0, atol=1e-12)
    for causal in (True, False):
        q1, k1, v1 = q[:, :, :1], k[:, :, :1], v[:, :, :1]
        O1, L1 = attn(np.ascontiguousarray(q1), np.ascontiguousarray(k1), np.ascontiguousarray(v1),
                      scale, causal)
        assert np.array_equal(O1, f64(v1))
        np.testing.assert_allclose(L1[:, :, 0], float(np.float32(scale)) * dots, rtol=0, atol=1e-12)


def pin_q_zero_mean(attn):
    """Q = 0 makes every score 0: O_i = mean(V_0..V_i) and LSE_i = ln(i+1) (causal);
    mean of all V and ln S without the mask.  GQA shape."""
    B, Hq, Hkv, S, D = 2, 4, 2, 23, 8
    q = np.zeros((B, Hq, S, D), np.uint16)  # +0.0 in bf16
    k = _rand((B, Hkv, S, D), 41, 1)
    v = _rand((B, Hkv, S, D), 41, 2)
    vf = np.repeat(f64(v), Hq // Hkv, axis=1)
    O, L = attn(q, k, v, 0.125, True)
    counts = np.arange(1, S + 1, dtype=np.float64)
    np.testing.assert_allclose(O, np.cumsum(vf, axis=2) / counts[None, None, :, None],
                               rtol=0, atol=1e-13)
    np.testing.assert_allclose(L, np.broadcast_to(np.log(counts), L.shape), rtol=0, atol=1e-13)
    O, L = attn(q, k, v, 0.125, False)
    np.testing.assert_allclose(O, np.broadcast_to(vf.mean(axis=2, keepdims=True), O.shape),
                               rtol=0, atol=1e-13)
    np.testing.assert_allclose(L, math.log(S), rtol=0, atol=1e-13)


def pin_key_shift(attn):
    """Adding one vector c to every key adds scale q_i.c to every score of row i:
    softmax is unchanged (O unchanged) and LSE_i grows by scale q_i.c."""
    rng = np.random.default_rng(51)
    B, H, S, D = 1, 2, 17, 8
    q = bits(_grid((B, H, S, D), rng, -2, 2, 0.125))
    k = _grid((B, H, S, D), rng, -2, 2, 0.125)
    c = _grid((D,), rng, -1, 1, 0.125)
    v = _rand((B, H, S, D), 51, 2)
    scale = 0.5
    for causal in (True, False):
        O0, L0 = attn(q, bits(k), v, scale, causal)
        O1, L1 = attn(q, bits(k + c), v, scale, causal)
        np.testing.assert_allclose(O1, O0, rtol=0, atol=1e-12)
        np.testing.assert_allclose(L1 - L0, scale * (f64(q) @ c), rtol=0, atol=1e-12)


def pin_value_linearity(attn):
    """O is affine in V with weights summing to 1: V = const gives O = const, and
    O(V1 + V2) = O(V1) + O(V2)."""
    rng = np.random.default_rng(61)
    B, H, S, D = 1, 2, 19, 8
    q = _rand((B, H, S, D), 61, 0)
    k = _rand((B, H, S, D), 61, 1)
    const = bits(np.broadcast_to(_grid((1, 1, 1, D), rng, -3, 3, 0.25), (B, H, S, D)))
    O, _ = attn(q, k, const, 0.35, True)
    np.testing.assert_allclose(O, f64(const), rtol=0, atol=1e-13)
    v1 = _grid((B, H, S, D), rng, -2, 2, 0.25)
    v2 = _grid((B, H, S, D), rng, -2, 2, 0.25)
    for causal in (True, False):
        Oa, _ = attn(q, k, bits(v1), 0.35, causal)
        Ob, _ = attn(q, k, bits(v2), 0.35, causal)
        Os, _ = attn(q, k, bits(v1 + v2), 0.35, causal)
        np.testing.assert_allclose(Os, Oa + Ob, rtol=0, atol=1e-12)


def pin_causality(attn):
    """Changing keys/values after position i leaves row i unchanged (exactly);
    the last causal row equals the unmasked last row."""
    B, H, S, D = 1, 2, 16, 8
    q, k, v = (_rand((B, H, S, D), 71, t) for t in range(3))
    O, L = attn(q, k, v, 0.3, True)
    cut = 6
    k2, v2 = k.copy(), v.copy()
    k2[:, :, cut + 1:] = _rand((B, H, S - cut - 1, D), 72, 1)
    v2[:, :, cut + 1:] = _rand((B, H, S - cut - 1, D), 72, 2)
    O2, L2 = attn(q, k2, v2, 0.3, True)
    assert np.array_equal(O2[:, :, :cut + 1], O[:, :, :cut + 1])
    assert np.array_equal(L2[:, :, :cut + 1], L[:, :, :cut + 1])
    assert not np.allclose(O2[:, :, cut + 1:], O[:, :, cut + 1:])
    On, Ln = attn(q, k, v, 0.3, False)
    np.testing.assert_allclose(O[:, :, -1], On[:, :, -1], rtol=0, atol=1e-14)
    np.testing.assert_allclose(L[:, :, -1], Ln[:, :, -1], rtol=0, atol=1e-14)
    assert not np.allclose(O[:, :, 0], On[:, :, 0])


def pin_heads_and_batches(attn):
    """GQA equals multi-head attention on key/value heads repeated in contiguous
    groups; batch entries are independent of each other."""
    B, Hq, Hkv, S, D = 3, 6, 2, 11, 8
    q = _rand((B, Hq, S, D), 81, 0)
    k = _rand((B, Hkv, S, D), 81, 1)
    v = _rand((B, Hkv, S, D), 81, 2)
    O, L = attn(q, k, v, 0.3, True)
    ke = np.ascontiguousarray(np.repeat(k, Hq // Hkv, axis=1))
    ve = np.ascontiguousarray(np.repeat(v, Hq // Hkv, axis=1))
    Oe, Le = attn(q, ke, ve, 0.3, True)
    assert np.array_equal(O, Oe) and np.array_equal(L, Le)
    for b in range(B):
        Ob, Lb = attn(np.ascontiguousarray(q[b:b + 1]), np.ascontiguousarray(k[b:b + 1]),
                      np.ascontiguousarray(v[b:b + 1]), 0.3, True)
        assert np.array_equal(Ob[0], O[b]) and np.array_equal(Lb[0], L[b])


def pin_large_magnitude(attn):
    """Scores in the thousands (Q x 1024) still give finite results equal to the
    library's float64 SDPA: the softmax must subtract the row maximum."""
    B, H, S, D = 1, 2, 24, 16
    q = _rand((B, H, S, D), 91, 0)
    k = _rand((B, H, S, D), 91, 1)
    v = _rand((B, H, S, D), 91, 2)
    q_big = float32_to_bf16_bits(bf16_bits_to_float32(q) * np.float32(1024.0))
    for causal in (True, False):
        O, L = attn(q_big, k, v, 0.25, causal)
        assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))
        np.testing.assert_allclose(O, _sdpa64(q_big, k, v, 0.25, causal), rtol=0, atol=1e-10)


def pin_worked_example(attn):
    """The hand-derived S = 3 example in tests/golden/worked_example_s3.json."""
    with open(os.path.join(GOLDEN, "worked_example_s3.json")) as f:
        ex = json.load(f)
    sh = ex["shape"]
    shp = (sh["B"], sh["Hq"], sh["S"], sh["D"])
    q = bits(np.array(ex["q"]).reshape(shp))
    k = bits(np.array(ex["k"]).reshape(shp))
    v = bits(np.array(ex["v"]).reshape(shp))
    env = {"e": math.e, "ln": math.log, "__builtins__": {}}

    def ev(s):
        return eval(s, env)  # expressions from the fixture, e.g. "1/(1+e)"

    O, L = attn(q, k, v, ex["scale"], True)
    exp_o = np.array([[ev(s) for s in row] for row in ex["causal"]["out"]])
    exp_l = np.array([ev(s) for s in ex["causal"]["lse"]])
    np.testing.assert_allclose(O[0, 0], exp_o, rtol=0, atol=1e-15)
    np.testing.assert_allclose(L[0, 0], exp_l, rtol=0, atol=1e-15)
    O, L = attn(q, k, v, ex["scale"], False)
    rows = ex["noncausal"]["rows"]
    exp_o = np.array([[ev(s) for s in row] for row in ex["noncausal"]["out"]])
    exp_l = np.array([ev(s) for s in ex["noncausal"]["lse"]])
    np.testing.assert_allclose(O[0, 0, rows], exp_o, rtol=0, atol=1e-15)
    np.testing.assert_allclose(L[0, 0, rows], exp_l, rtol=0, atol=1e-15)


ALL_PINS = [
    pin_sdpa_library,
    pin_attention_matrix,
    pin_row0_and_s1,
    pin_q_zero_mean,
    pin_key_shift,
    pin_value_linearity,
    pin_causality,
    pin_heads_and_batches,
    pin_large_magnitude,
    pin_worked_example,
]


# ---------------------------------------------------------------------------
# FP8 E4M3 inputs (the oracle's second entry point).  The callable for these
# pins is ``attn8(q_codes, k_codes, v_codes, scale, descales, causal)`` and
# ``decode(codes)``.
def _e4m3_codes(shape, seed, stream, sigma=1.0):
    """Random E4M3 codes from N(0, sigma^2) values, quantised by torch (a library
    conversion, independent of the oracle's decoding)."""
    x = bf16_bits_to_float32(gaussian_bf16(shape, seed, stream, sigma))
    t = torch.from_numpy(np.ascontiguousarray(x)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


def _torch_e4m3(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64)


def pin_e4m3_decode(decode):
    """All 256 codes decode as torch's float8_e4m3fn (NaN codes as NaN)."""
    codes = np.arange(256, dtype=np.uint8)
    ref = _torch_e4m3(codes).numpy()
    got = decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


def pin_e4m3_sdpa_library(attn8):
    """FP8 inputs with non-trivial descales equal torch's float64 SDPA on the
    dequantised tensors (causal and not, GQA)."""
    B, Hq, Hkv, S, D = 2, 4, 2, 33, 16
    q, k, v = (_e4m3_codes((B, H, S, D), 111, t) for t, H in ((0, Hq), (1, Hkv), (2, Hkv)))
    ds = tuple(float(np.float32(x)) for x in (0.37, 1.9, 0.61))  # descales travel as fp32
    scale = 1.0 / math.sqrt(D)
    for causal in (True, False):
        O, L = attn8(q, k, v, scale, ds, causal)
        qf, kf, vf = (_torch_e4m3(c) * d for c, d in zip((q, k, v), ds))
        kf = kf.repeat_interleave(Hq // Hkv, dim=1)
        vf = vf.repeat_interleave(Hq // Hkv, dim=1)
        ref = F.scaled_dot_product_attention(qf, kf, vf, is_causal=causal,
                                             scale=float(np.float32(scale))).numpy()
        np.testing.assert_allclose(O, ref, rtol=0, atol=1e-12)
        # LSE from its definition on the dequantised scores (a library logsumexp)
        sc = torch.einsum("bhid,bhjd->bhij", qf, kf) * float(np.float32(scale))
        if causal:
            sc = sc.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
        np.testing.assert_allclose(L, torch.logsumexp(sc, dim=-1).numpy(), rtol=0, atol=1e-12)


def pin_e4m3_matches_bf16_path(attn8, attn):
    """Every E4M3 value is exact in bf16, so with unit descales the FP8 entry equals
    the bf16 entry on the same values; power-of-two descales scale exactly."""
    B, H, S, D = 1, 3, 20, 8
    q, k, v = (_e4m3_codes((B, H, S, D), 121, t) for t in range(3))
    to_bf16 = lambda c, d: float32_to_bf16_bits(  # noqa: E731
        (_torch_e4m3(c) * d).to(torch.float32).numpy())
    for ds in ((1.0, 1.0, 1.0), (2.0, 0.25, 8.0)):
        O8, L8 = attn8(q, k, v, 0.3, ds, True)
        O, L = attn(to_bf16(q, ds[0]), to_bf16(k, ds[1]), to_bf16(v, ds[2]), 0.3, True)
        assert np.array_equal(O8, O) and np.array_equal(L8, L)


E4M3_PINS = [pin_e4m3_decode, pin_e4m3_sdpa_library, pin_e4m3_matches_bf16_path]


# ---------------------------------------------------------------------------
# Block masks (the oracle's masked entry).  attnm(q, k, v, scale, mask, causal).
def _expand_block_mask(mask, Hq, S, causal):
    """Element mask [Hq, S, S] (True = visible) from a [Hm, nt, nt] block mask."""
    m = torch.from_numpy(np.ascontiguousarray(mask)).bool()
    m = m.repeat_interleave(128, dim=1).repeat_interleave(128, dim=2)[:, :S, :S]
    m = m.expand(Hq, S, S)
    if causal:
        m = m & torch.ones(S, S, dtype=torch.bool).tril()
    return m


def pin_block_mask_library(attnm):
    """Random block masks (shared and per head, causal and not, GQA) against torch's
    float64 SDPA with the expanded boolean mask; rows that see no key are 0 there
    (its safe softmax) and must have LSE = -inf; other LSEs against logsumexp."""
    rng = np.random.default_rng(131)
    B, Hq, Hkv, S, D = 2, 4, 2, 300, 8
    nt = 3
    q, k, v = (_rand((B, H, S, D), 131, t) for t, H in ((0, Hq), (1, Hkv), (2, Hkv)))
    scale = 0.35
    for hm, causal in ((1, True), (Hq, False), (Hq, True)):
        mask = (rng.random((hm, nt, nt)) < 0.6).astype(np.uint8)
        mask[0, 2, :] = 0  # query tile 2 of head 0 sees nothing
        O, L = attnm(q, k, v, scale, mask, causal)
        em = _expand_block_mask(mask, Hq, S, causal)
        qf = torch.from_numpy(f64(q))
        kf = torch.from_numpy(f64(k)).repeat_interleave(Hq // Hkv, dim=1)
        vf = torch.from_numpy(f64(v)).repeat_interleave(Hq // Hkv, dim=1)
        sc32 = float(np.float32(scale))
        ref = F.scaled_dot_product_attention(qf, kf, vf, attn_mask=em, scale=sc32).numpy()
        np.testing.assert_allclose(O, ref, rtol=0, atol=1e-12)
        sc = torch.einsum("bhid,bhjd->bhij", qf, kf) * sc32
        lse_ref = torch.logsumexp(sc.masked_fill(~em, float("-inf")), dim=-1).numpy()
        none = ~em.any(dim=-1).numpy()  # [Hq, S]
        assert none.any()
        assert np.all(np.isneginf(L[:, none])) and np.all(O[:, none] == 0.0)
        np.testing.assert_allclose(L[:, ~none], lse_ref[:, ~none], rtol=0, atol=1e-12)


def pin_block_mask_all_ones(attnm, attn):
    """An all-ones block mask changes nothing."""
    B, H, S, D = 1, 2, 200, 8
    q, k, v = (_rand((B, H, S, D), 141, t) for t in range(3))
    for causal in (True, False):
        Om, Lm = attnm(q, k, v, 0.3, np.ones((1, 2, 2), np.uint8), causal)
        O, L = attn(q, k, v, 0.3, causal)
        assert np.array_equal(Om, O) and np.array_equal(Lm, L)


MASK_PINS = [pin_block_mask_library, pin_block_mask_all_ones]


# ---------------------------------------------------------------- gradients
# Each takes ``bwd(q, k, v, dout, scale, causal, kv_heads=None)`` returning
# (dQ, dK, dV, delta) in float64 (bf16 bit patterns or float64 inputs).

def _loss_grad_fd(fwd64, q, k, v, dout, scale, causal, h=1e-5):
    """Central differences of L = sum(dout * O) with respect to every element
    of q, k and v, each from two calls of the forward oracle on float64 inputs."""
    def loss(qq, kk, vv):
        return float(np.sum(dout * fwd64(qq, kk, vv, scale, causal)[0]))
    grads = []
    for which in range(3):
        base = [q, k, v]
        g = np.zeros_like(base[which])
        for idx in np.ndindex(g.shape):
            plus = [x.copy() for x in base]
            minus = [x.copy() for x in base]
            plus[which][idx] += h
            minus[which][idx] -= h
            g[idx] = (loss(*plus) - loss(*minus)) / (2 * h)
        grads.append(g)
    return grads


def pin_bwd_finite_differences(bwd, fwd64):
    """Gradients against central differences of the forward oracle (float64
    inputs, step 1e-5: truncation ~1e-10), GQA, causal and not; delta against
    sum_d dO_id O_id from the forward output."""
    rng = np.random.default_rng(151)
    B, Hq, Hkv, S, D = 1, 2, 1, 6, 3
    q, dout = rng.standard_normal((B, Hq, S, D)), rng.standard_normal((B, Hq, S, D))
    k, v = rng.standard_normal((B, Hkv, S, D)), rng.standard_normal((B, Hkv, S, D))
    for causal in (True, False):
        dq, dk, dv, delta = bwd(q, k, v, dout, 0.6, causal)
        fq, fk, fv = _loss_grad_fd(fwd64, q, k, v, dout, 0.6, causal)
        for name, a, b in (("dQ", dq, fq), ("dK", dk, fk), ("dV", dv, fv)):
            err = float(np.max(np.abs(a - b)))
            assert err < 1e-7, f"{name} vs finite differences: {err:.2e} (causal={causal})"
        O = fwd64(q, k, v, 0.6, causal)[0]
        assert np.max(np.abs(delta - np.sum(dout * O, axis=-1))) < 1e-12


def pin_bwd_torch_autograd(bwd):
    """Gradients against torch's float64 autograd through scaled_dot_product_attention
    on CPU (key/value heads expanded with repeat_interleave, whose backward sums
    the group), causal and not, several tiles and a ragged tail."""
    B, Hq, Hkv, S, D = 2, 4, 2, 150, 16
    q, k, v = (_rand((B, H, S, D), 161, t) for t, H in ((0, Hq), (1, Hkv), (2, Hkv)))
    dout = _rand((B, Hq, S, D), 161, 3)
    scale = 0.3
    G = Hq // Hkv
    for causal in (True, False):
        dq, dk, dv, delta = bwd(q, k, v, dout, scale, causal)
        tq, tk, tv = (torch.from_numpy(f64(x)).requires_grad_() for x in (q, k, v))
        o = F.scaled_dot_product_attention(tq, tk.repeat_interleave(G, 1), tv.repeat_interleave(G, 1),
                                           is_causal=causal, scale=float(np.float32(scale)))
        o.backward(torch.from_numpy(f64(dout)))
        for name, a, t in (("dQ", dq, tq), ("dK", dk, tk), ("dV", dv, tv)):
            ref = t.grad.numpy()
            err = float(np.max(np.abs(a - ref)))
            assert err <= 1e-12 * max(1.0, float(np.max(np.abs(ref)))), f"{name}: {err:.2e}"
        ref_delta = np.sum(f64(dout) * o.detach().numpy(), axis=-1)
        assert np.max(np.abs(delta - ref_delta)) < 1e-12


def pin_bwd_closed_forms(bwd):
    """Causal row 0 attends to key 0 alone (weight exactly 1), so dQ_0 = 0
    exactly.  Weights sum to 1 in every row, so the dV rows sum to the dO rows
    of the group and the dK rows sum to 0.  With Q = 0 the causal weights are
    1/(i+1), so dV_j = sum_{i>=j} dO_i / (i+1)."""
    B, Hq, Hkv, S, D = 1, 4, 2, 90, 8
    q, k, v = (_rand((B, H, S, D), 171, t) for t, H in ((0, Hq), (1, Hkv), (2, Hkv)))
    dout = _rand((B, Hq, S, D), 171, 3)
    dq, dk, dv, _ = bwd(q, k, v, dout, 0.4, True)
    assert np.all(dq[:, :, 0, :] == 0.0), "causal row 0 must have dQ = 0"
    d64 = f64(dout).reshape(B, Hkv, Hq // Hkv, S, D)
    assert np.max(np.abs(dv.sum(axis=2) - d64.sum(axis=(2, 3)))) < 1e-11
    assert np.max(np.abs(dk.sum(axis=2))) < 1e-11
    qz = bits(np.zeros((1, 1, S, D)))
    _, _, dvz, _ = bwd(qz, k[:, :1], v[:, :1], dout[:, :1], 0.4, True)
    do1 = f64(dout[0, 0])
    want = np.array([sum(do1[i] / (i + 1) for i in range(j, S)) for j in range(S)])
    assert np.max(np.abs(dvz[0, 0] - want)) < 1e-12


def pin_bwd_invariants(bwd):
    """Adding a constant vector to every key leaves the output unchanged as a
    function of Q, K, V, so the gradients do not change; the gradients are
    linear in dO; a subset of key/value heads gives exactly those heads."""
    B, Hq, Hkv, S, D = 2, 4, 2, 70, 8
    rng = np.random.default_rng(181)
    q = bits(_grid((B, Hq, S, D), rng, -2, 2, 0.25))
    k = bits(_grid((B, Hkv, S, D), rng, -2, 2, 0.25))
    v = bits(_grid((B, Hkv, S, D), rng, -2, 2, 0.25))
    d1 = bits(_grid((B, Hq, S, D), rng, -2, 2, 0.25))
    d2 = bits(_grid((B, Hq, S, D), rng, -2, 2, 0.25))
    c = bits(_grid((D,), rng, -1, 1, 0.25))
    ks = bits(f64(k) + f64(c))
    for causal in (True, False):
        g = bwd(q, k, v, d1, 0.5, causal)
        gs = bwd(q, ks, v, d1, 0.5, causal)
        for a, b in zip(g[:3], gs[:3]):
            assert np.max(np.abs(a - b)) < 1e-11, "key shift changed a gradient"
        g2 = bwd(q, k, v, d2, 0.5, causal)
        g12 = bwd(q, k, v, bits(f64(d1) + f64(d2)), 0.5, causal)
        for a, b, s in zip(g[:3], g2[:3], g12[:3]):
            assert np.max(np.abs(a + b - s)) < 1e-11, "gradients not linear in dO"
        sub = bwd(q, k, v, d1, 0.5, causal, kv_heads=[3, 0])
        G = Hq // Hkv
        dq = g[0].reshape(B * Hkv, G, S, D)
        assert np.array_equal(sub[0], dq[[3, 0]])
        assert np.array_equal(sub[1], g[1].reshape(B * Hkv, S, D)[[3, 0]])
        assert np.array_equal(sub[2], g[2].reshape(B * Hkv, S, D)[[3, 0]])


BWD_PINS = [pin_bwd_torch_autograd, pin_bwd_closed_forms, pin_bwd_invariants]
# (the block-masked gradient pins are defined below; see BWD_MASK_PINS)


# ---------------------------------------------------------------- dropout
# ``attnd(q, k, v, scale, p8, seed, offset, causal, rows=None)`` -> (O, LSE).

# The Random123 known-answer list (Salmon et al.'s distribution of the
# generator), philox4x32 with 10 rounds: counter words 0..3, key words 0..1 ->
# output words 0..3.
PHILOX4X32_10_KNOWN_ANSWERS = [
    ((0x00000000, 0x00000000, 0x00000000, 0x00000000), (0x00000000, 0x00000000),
     (0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8)),
    ((0xffffffff, 0xffffffff, 0xffffffff, 0xffffffff), (0xffffffff, 0xffffffff),
     (0x408f276d, 0x41c83b0e, 0xa20bc7c6, 0x6d5451fd)),
    ((0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344), (0xa4093822, 0x299f31d0),
     (0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1)),
]


def numpy_philox4x32(ctr, key):
    """Philox4x32-10 of counters ``ctr`` ([n, 4] uint32 words) under ``key``
    ([2] or [n, 2]), vectorised in numpy's uint64 arithmetic: a test-side
    generator, itself checked against the published known answers
    (pin_test_generator_known_answers) and Triton's implementation."""
    x = np.array(ctr, dtype=np.uint64).reshape(-1, 4)
    k = np.broadcast_to(np.array(key, dtype=np.uint64).reshape(-1, 2), (x.shape[0], 2)).copy()
    lo = np.uint64(0xFFFFFFFF)
    for _ in range(10):
        p0 = np.uint64(0xD2511F53) * x[:, 0]  # both factors < 2^32: exact in uint64
        p1 = np.uint64(0xCD9E8D57) * x[:, 2]
        x = np.stack([(p1 >> np.uint64(32)) ^ x[:, 1] ^ k[:, 0], p1 & lo,
                      (p0 >> np.uint64(32)) ^ x[:, 3] ^ k[:, 1], p0 & lo], axis=1)
        k = (k + np.array([0x9E3779B9, 0xBB67AE85], dtype=np.uint64)) & lo
    return x.astype(np.uint32)


def pin_test_generator_known_answers():
    for ctr, key, want in PHILOX4X32_10_KNOWN_ANSWERS:
        assert [int(x) for x in numpy_philox4x32([ctr], key)[0]] == list(want)


def keep_table(bh, S, p8, seed, offset):
    """[S, S] booleans: is key j of query i kept?  The documented mapping --
    byte (j mod 16) of Philox4x32-10(counter {j/16, i, bh, offset}, key
    {seed mod 2^32, seed / 2^32}), little-endian words in order, kept when
    >= p8 -- written from the definition with the test-side generator."""
    nblk = (S + 15) // 16
    i, blk = np.meshgrid(np.arange(S), np.arange(nblk), indexing="ij")
    ctr = np.stack([blk.ravel(), i.ravel(), np.full(i.size, bh), np.full(i.size, offset)], axis=1)
    by = numpy_philox4x32(ctr, [seed & 0xFFFFFFFF, seed >> 32]).view(np.uint8).reshape(S, nblk * 16)
    return by[:, :S] >= p8


TRITON_PHILOX = r"""
import json, sys
import torch, triton, triton.language as tl

@triton.jit
def blocks(out_ptr, c_ptr, seed, N: tl.constexpr):
    i = tl.arange(0, N)
    a, b, c, d = tl.philox(seed, tl.load(c_ptr + 4 * i), tl.load(c_ptr + 4 * i + 1),
                           tl.load(c_ptr + 4 * i + 2), tl.load(c_ptr + 4 * i + 3))
    tl.store(out_ptr + 4 * i, a)
    tl.store(out_ptr + 4 * i + 1, b)
    tl.store(out_ptr + 4 * i + 2, c)
    tl.store(out_ptr + 4 * i + 3, d)

res = []
for seed, ctrs in json.loads(sys.stdin.read()):
    c = torch.tensor(ctrs, dtype=torch.int64).to(torch.int32).reshape(-1)
    out = torch.zeros(c.numel(), dtype=torch.int32)
    blocks[(1,)](out, c, seed, N=len(ctrs))
    res.append([x & 0xFFFFFFFF for x in out.tolist()])
print(json.dumps(res))
"""


def triton_philox4x32(cases):
    """Philox4x32-10 blocks from Triton's own tl.philox (a library routine, key
    {seed mod 2^32, seed / 2^32}), run by its CPU interpreter in a subprocess;
    ``cases`` = [(seed, [[c0, c1, c2, c3], ...]), ...] with a power-of-two
    count of counters each.  None when Triton's interpreter is unavailable."""
    import json
    import os
    import subprocess
    import sys
    try:
        import triton  # noqa: F401
    except ImportError:
        return None
    env = dict(os.environ, TRITON_INTERPRET="1")
    res = subprocess.run([sys.executable, "-c", TRITON_PHILOX], input=json.dumps(cases), env=env,
                         capture_output=True, text=True, timeout=300)
    if res.returncode != 0:
        return None
    return [np.array(r, dtype=np.uint64).reshape(-1, 4) for r in json.loads(res.stdout)]


def pin_philox_known_answers(philox):
    """The oracle's Philox4x32-10 block gives the published known answers."""
    for ctr, key, want in PHILOX4X32_10_KNOWN_ANSWERS:
        assert [int(x) for x in philox(ctr, key)] == list(want)


def pin_philox_library(philox):
    """The oracle's Philox4x32-10 block equals the test-side generator and
    Triton's tl.philox (when its interpreter runs here) for assorted counters
    and keys."""
    rng = np.random.default_rng(191)
    cases = []
    for _ in range(8):
        seed = int(rng.integers(0, 2**63)) * 2 + int(rng.integers(0, 2))
        ctrs = [[int(x) for x in rng.integers(0, 2**32, 4, dtype=np.uint64)] for _ in range(4)]
        cases.append((seed, ctrs))
        key = [seed & 0xFFFFFFFF, seed >> 32]
        for c in ctrs:
            assert np.array_equal(philox(c, key).astype(np.uint64),
                                  numpy_philox4x32([c], key)[0].astype(np.uint64))
    lib = triton_philox4x32(cases)
    if lib is not None:
        for (seed, ctrs), blocks in zip(cases, lib):
            key = [seed & 0xFFFFFFFF, seed >> 32]
            for c, want in zip(ctrs, blocks):
                assert np.array_equal(philox(c, key).astype(np.uint64), want)


def pin_dropout_mask_closed_form(attnd, attn):
    """V = identity rows turns O rows into the weights: with dropout each must be
    the undropped weight times keep(i, j) * 256/(256-p8), keep from the
    documented byte mapping over the test-side Philox4x32-10 (counter word 2 =
    b * H + h, so two batches draw different decisions; counter word 3 = the
    offset; a seed above 2^32 puts both key words to use); the LSE is
    unchanged."""
    B, H, S, D = 2, 2, 70, 128
    q, k = _rand((B, H, S, D), 201, 0), _rand((B, H, S, D), 201, 1)
    v = bits(np.broadcast_to(np.eye(S, D), (B, H, S, D)))
    p8, seed, offset = 77, 0x5eed0001234abcd, 99
    for causal in (True, False):
        O, L = attnd(q, k, v, 0.2, p8, seed, offset, causal)
        P, L0 = attn(q, k, v, 0.2, causal)
        assert np.array_equal(L, L0), "dropout changed the LSE"
        for b in range(B):
            for h in range(H):
                keep = keep_table(b * H + h, S, p8, seed, offset)
                want = P[b, h, :, :S] * keep * (256.0 / (256 - p8))
                assert np.max(np.abs(O[b, h, :, :S] - want)) < 1e-15


def pin_dropout_rate_and_identity(attnd, attn):
    """p8 = 0 is no dropout (bit for bit); with p8 = 64 a quarter of the weights
    are dropped (within five binomial standard deviations)."""
    B, H, S, D = 1, 4, 128, 128
    q, k = _rand((B, H, S, D), 211, 0), _rand((B, H, S, D), 211, 1)
    v = bits(np.broadcast_to(np.eye(S, D), (B, H, S, D)))
    O0, L0 = attnd(q, k, v, 0.1, 0, 5, 6, False)
    O, L = attn(q, k, v, 0.1, False)
    assert np.array_equal(O0, O) and np.array_equal(L0, L)
    Od, _ = attnd(q, k, v, 0.1, 64, 5, 6, False)
    dropped = float(np.mean(Od == 0.0))
    n = Od.size
    assert abs(dropped - 0.25) < 5 * math.sqrt(0.25 * 0.75 / n), dropped


DROPOUT_PINS = [pin_dropout_mask_closed_form, pin_dropout_rate_and_identity]


# ---------------------------------------------------------------- output projection
# ``proj(o, w, bias)`` -> Y [B, S, E] float64.

def pin_proj_library(proj):
    """Against torch's float64 linear on the concatenated heads (torch.cat of the
    per-head outputs along the feature axis, the form the pages' layer uses)."""
    B, H, S, D, E = 2, 3, 20, 16, 40
    o = _rand((B, H, S, D), 221, 0)
    w = _rand((E, H * D), 221, 1)
    bias = np.random.default_rng(221).standard_normal(E)
    Y = proj(o, w, bias)
    heads = [torch.from_numpy(f64(o[:, h])) for h in range(H)]       # [B, S, D] each
    cat = torch.cat(heads, dim=-1)                                     # [B, S, H*D]
    ref = F.linear(cat, torch.from_numpy(f64(w)), torch.from_numpy(bias)).numpy()
    assert np.max(np.abs(Y - ref)) < 1e-12


def pin_proj_selection(proj):
    """W picking one input feature per output (W[e, h*D + d] = 1): Y[b, s, e] is
    exactly O[b, h, s, d]; with O = 0 the output is the bias."""
    B, H, S, D = 1, 4, 9, 8
    o = _rand((B, H, S, D), 231, 0)
    picks = [(3, 5), (0, 0), (2, 7), (1, 2), (3, 0), (0, 6), (2, 2), (1, 7)]
    w = np.zeros((len(picks), H * D), dtype=np.float32)
    for e, (h, d) in enumerate(picks):
        w[e, h * D + d] = 1.0
    Y = proj(o, bits(w), None)
    for e, (h, d) in enumerate(picks):
        assert np.array_equal(Y[0, :, e], f64(o[0, h, :, d]))
    bias = np.arange(len(picks), dtype=np.float64) - 2.5
    Yb = proj(bits(np.zeros((B, H, S, D))), bits(w), bias)
    assert np.array_equal(Yb, np.broadcast_to(bias, Yb.shape))


PROJ_PINS = [pin_proj_library, pin_proj_selection]


def pin_bwd_masked_library(bwdm):
    """Block-masked gradients against torch's float64 autograd through SDPA with the
    expanded boolean mask; a query tile that sees no key has zero gradients on
    both sides (torch's safe softmax)."""
    B, Hq, Hkv, S, D = 1, 4, 2, 300, 8
    q, k, v = (_rand((B, H, S, D), 241, t) for t, H in ((0, Hq), (1, Hkv), (2, Hkv)))
    dout = _rand((B, Hq, S, D), 241, 3)
    rng = np.random.default_rng(241)
    nt = 3
    G = Hq // Hkv
    for hm, causal in ((Hq, True), (1, False), (Hq, False)):
        mask = (rng.random((hm, nt, nt)) < 0.7).astype(np.uint8)
        mask[0, 2, :] = 0
        dq, dk, dv, _ = bwdm(q, k, v, dout, 0.5, causal, mask)
        allowed = _expand_block_mask(mask, Hq, S, causal)  # [Hq, S, S], True = visible
        tq, tk, tv = (torch.from_numpy(f64(x)).requires_grad_() for x in (q, k, v))
        o = F.scaled_dot_product_attention(tq, tk.repeat_interleave(G, 1), tv.repeat_interleave(G, 1),
                                           attn_mask=allowed[None], scale=float(np.float32(0.5)))
        o.backward(torch.from_numpy(f64(dout)))
        for name, a, t in (("dQ", dq, tq), ("dK", dk, tk), ("dV", dv, tv)):
            ref = t.grad.numpy()
            assert not np.isnan(ref).any()
            assert np.max(np.abs(a - ref)) <= 1e-12 * max(1.0, float(np.max(np.abs(ref)))), name
        assert np.all(dq[0, 0, 256:] == 0.0)


def pin_bwd_masked_all_ones(bwdm, bwd):
    """The all-ones block mask gives the unmasked gradients bit for bit."""
    B, H, S, D = 1, 2, 200, 8
    q, k, v = (_rand((B, H, S, D), 251, t) for t in range(3))
    dout = _rand((B, H, S, D), 251, 3)
    for causal in (True, False):
        a = bwdm(q, k, v, dout, 0.3, causal, np.ones((1, 2, 2), np.uint8))
        b = bwd(q, k, v, dout, 0.3, causal)
        assert all(np.array_equal(x, y) for x, y in zip(a, b))


BWD_MASK_PINS = [pin_bwd_masked_library]


# ---------------------------------------------------------------- element masks
# ``attnk(q, k, v, scale, keep_bits, causal, block_mask=None)`` returns (O, LSE);
# keep_bits uint8 [Hm, S, 16 * ceil(S/128)], bit j % 8 of byte j / 8 of row i
# keeps key j for query i.

def _keep_rows(S):
    return 16 * ((S + 127) // 128)


def _keep_to_bool(bits, S):
    """Element mask [Hm, S, S] (True = kept) unpacked bit by bit, independently of
    the packing helper the tests use to build masks."""
    bits = np.asarray(bits, dtype=np.uint8)
    j = np.arange(S)
    return ((bits[:, :, j // 8] >> (j % 8)) & 1).astype(bool)


def pin_keep_library(attnk):
    """Random element masks (shared and per head, causal and not, GQA, with and
    without a block mask on top) against torch's float64 SDPA with the same boolean
    mask; rows that see no key are 0 there and must have LSE = -inf."""
    rng = np.random.default_rng(311)
    B, Hq, Hkv, S, D = 2, 4, 2, 300, 8
    q, k, v = (_rand((B, H, S, D), 311, t) for t, H in ((0, Hq), (1, Hkv), (2, Hkv)))
    scale = 0.35
    sc32 = float(np.float32(scale))
    qf = torch.from_numpy(f64(q))
    kf = torch.from_numpy(f64(k)).repeat_interleave(Hq // Hkv, dim=1)
    vf = torch.from_numpy(f64(v)).repeat_interleave(Hq // Hkv, dim=1)
    for hm, causal, density, with_block in ((1, True, 0.5, False), (Hq, False, 0.3, False),
                                            (Hq, True, 0.8, True), (1, False, 0.6, True)):
        keep = rng.random((hm, S, S)) < density
        keep[0, 7, :] = False  # query 7 of head 0 sees nothing
        bits = np.zeros((hm, S, _keep_rows(S)), np.uint8)
        for jj in range(S):
            bits[:, :, jj // 8] |= (keep[:, :, jj].astype(np.uint8) << (jj % 8))
        bm = (rng.random((hm, 3, 3)) < 0.7).astype(np.uint8) if with_block else None
        O, L = attnk(q, k, v, scale, bits, causal, bm)
        em = torch.from_numpy(keep).expand(Hq, S, S)
        if bm is not None:
            em = em & _expand_block_mask(bm, Hq, S, False)
        if causal:
            em = em & torch.ones(S, S, dtype=torch.bool).tril()
        ref = F.scaled_dot_product_attention(qf, kf, vf, attn_mask=em, scale=sc32).numpy()
        np.testing.assert_allclose(O, ref, rtol=0, atol=1e-12)
        sc = torch.einsum("bhid,bhjd->bhij", qf, kf) * sc32
        lse_ref = torch.logsumexp(sc.masked_fill(~em, float("-inf")), dim=-1).numpy()
        none = ~em.any(dim=-1).numpy()
        assert none[0, 7]
        assert np.all(np.isneginf(L[:, none])) and np.all(O[:, none] == 0.0)
        np.testing.assert_allclose(L[:, ~none], lse_ref[:, ~none], rtol=0, atol=1e-12)


def pin_keep_selects_one_key(attnk):
    """Bytes written by hand: query i keeping only key j gives O_i = V_j exactly and
    LSE_i = the scaled score q_i . k_j (pins the bit order, the byte and row
    offsets and the per-head indexing of the element mask)."""
    B, H, S, D = 1, 2, 260, 8
    q, k, v = (_rand((B, H, S, D), 321, t) for t in range(3))
    R = _keep_rows(S)
    picks = [(0, 0, 0), (0, 5, 3), (1, 200, 137), (1, 259, 258), (0, 130, 9), (1, 17, 16)]
    bits = np.zeros((H, S, R), np.uint8)
    for h, i, j in picks:
        bits[h, i, j // 8] = np.uint8(1 << (j % 8))
    O, L = attnk(q, k, v, 0.25, bits, False, None)
    for h, i, j in picks:
        assert np.array_equal(O[0, h, i], f64(v[0, h, j]))
        s = float(np.dot(f64(q[0, h, i]), f64(k[0, h, j]))) * float(np.float32(0.25))
        assert abs(L[0, h, i] - s) <= 1e-12 * max(1.0, abs(s))
    others = np.ones((H, S), bool)
    for h, i, _ in picks:
        others[h, i] = False
    assert np.all(O[0][others] == 0.0) and np.all(np.isneginf(L[0][others]))


def pin_keep_equals_block_mask(attnk, attnm):
    """An element mask that keeps exactly the pairs of a block mask gives the
    block-masked result bit for bit; the all-ones element mask gives the unmasked one."""
    rng = np.random.default_rng(331)
    B, H, S, D = 1, 2, 300, 8
    q, k, v = (_rand((B, H, S, D), 331, t) for t in range(3))
    bm = (rng.random((H, 3, 3)) < 0.6).astype(np.uint8)
    keep = np.repeat(np.repeat(bm, 128, axis=1), 128, axis=2)[:, :S, :S].astype(bool)
    bits = np.zeros((H, S, _keep_rows(S)), np.uint8)
    for jj in range(S):
        bits[:, :, jj // 8] |= (keep[:, :, jj].astype(np.uint8) << (jj % 8))
    for causal in (True, False):
        Ok, Lk = attnk(q, k, v, 0.3, bits, causal, None)
        Om, Lm = attnm(q, k, v, 0.3, bm, causal)
        assert np.array_equal(Ok, Om) and np.array_equal(Lk, Lm)
        ones = np.full((1, S, _keep_rows(S)), 0xFF, np.uint8)
        Oa, La = attnk(q, k, v, 0.3, ones, causal, None)
        Om1, Lm1 = attnm(q, k, v, 0.3, np.ones((1, 3, 3), np.uint8), causal)
        assert np.array_equal(Oa, Om1) and np.array_equal(La, Lm1)
        assert np.array_equal(_keep_to_bool(bits, S), keep)


KEEP_PINS = [pin_keep_library, pin_keep_selects_one_key]


def pin_bwd_keep_library(bwdk):
    """Element-masked gradients against torch's float64 autograd through SDPA with
    the same boolean mask (a row that sees no key has zero gradients on both sides)."""
    B, Hq, Hkv, S, D = 1, 4, 2, 300, 8
    q, k, v = (_rand((B, H, S, D), 341, t) for t, H in ((0, Hq), (1, Hkv), (2, Hkv)))
    dout = _rand((B, Hq, S, D), 341, 3)
    rng = np.random.default_rng(341)
    G = Hq // Hkv
    for hm, causal, density in ((Hq, True, 0.6), (1, False, 0.4)):
        keep = rng.random((hm, S, S)) < density
        keep[0, 11, :] = False
        bits = np.zeros((hm, S, _keep_rows(S)), np.uint8)
        for jj in range(S):
            bits[:, :, jj // 8] |= (keep[:, :, jj].astype(np.uint8) << (jj % 8))
        dq, dk, dv, _ = bwdk(q, k, v, dout, 0.5, causal, bits)
        em = torch.from_numpy(keep).expand(Hq, S, S)
        if causal:
            em = em & torch.ones(S, S, dtype=torch.bool).tril()
        tq, tk, tv = (torch.from_numpy(f64(x)).requires_grad_() for x in (q, k, v))
        o = F.scaled_dot_product_attention(tq, tk.repeat_interleave(G, 1), tv.repeat_interleave(G, 1),
                                           attn_mask=em[None], scale=float(np.float32(0.5)))
        o.backward(torch.from_numpy(f64(dout)))
        for name, a, t in (("dQ", dq, tq), ("dK", dk, tk), ("dV", dv, tv)):
            ref = t.grad.numpy()
            assert not np.isnan(ref).any()
            assert np.max(np.abs(a - ref)) <= 1e-12 * max(1.0, float(np.max(np.abs(ref)))), name
        assert np.all(dq[0, 0, 11] == 0.0)


BWD_KEEP_PINS = [pin_bwd_keep_library]


def pin_bwd_dropout_autograd(bwdd):
    """Gradients with dropout against torch's float64 autograd of
    O = ((softmax of the masked scores) * Z * 256/(256-p8)) V, Z the keep table
    written from the documented byte mapping over the test-side Philox4x32-10; and p8 = 0
    gives the gradients without dropout bit for bit.  Two batches, so the keep
    table's counter carries the flat batch * head index."""
    B, Hq, Hkv, S, D = 2, 4, 2, 70, 8
    q, k, v = (_rand((B, H, S, D), 261, t) for t, H in ((0, Hq), (1, Hkv), (2, Hkv)))
    dout = _rand((B, Hq, S, D), 261, 3)
    G = Hq // Hkv
    p8, seed, offset = 51, 0xBEEF, 7
    s = 256.0 / (256 - p8)
    Z = torch.from_numpy(np.stack([np.stack([keep_table(b * Hq + h, S, p8, seed, offset) for h in range(Hq)])
                                   for b in range(B)]).astype(np.float64))
    for causal in (True, False):
        dq, dk, dv, delta = bwdd(q, k, v, dout, 0.4, causal, (p8, seed, offset))
        tq, tk, tv = (torch.from_numpy(f64(x)).requires_grad_() for x in (q, k, v))
        sc = torch.einsum("bhid,bhjd->bhij", tq, tk.repeat_interleave(G, 1)) * float(np.float32(0.4))
        if causal:
            sc = sc.masked_fill(~torch.ones(S, S, dtype=torch.bool).tril(), float("-inf"))
        o = torch.einsum("bhij,bhjd->bhid", torch.softmax(sc, dim=-1) * Z * s, tv.repeat_interleave(G, 1))
        o.backward(torch.from_numpy(f64(dout)))
        for name, a, t in (("dQ", dq, tq), ("dK", dk, tk), ("dV", dv, tv)):
            ref = t.grad.numpy()
            assert np.max(np.abs(a - ref)) <= 1e-12 * max(1.0, float(np.max(np.abs(ref)))), name
        want_delta = np.sum(f64(dout) * o.detach().numpy(), axis=-1)
        assert np.max(np.abs(delta - want_delta)) <= 1e-12 * max(1.0, float(np.max(np.abs(want_delta))))
        a0 = bwdd(q, k, v, dout, 0.4, causal, (0, seed, offset))
        b0 = bwdd(q, k, v, dout, 0.4, causal, None)
        assert all(np.array_equal(x, y) for x, y in zip(a0, b0))


BWD_DROPOUT_PINS = [pin_bwd_dropout_autograd]


# ---------------------------------------------------------------- combined variants
# ``attnx(q, k, v, scale, causal, descales=None, block_mask=None, keep_bits=None,
# dropout=None)`` and ``bwdx(q, k, v, dout, scale, causal, block_mask, keep_bits, dropout)``.

def _combo_inputs(seed, S=200, Hq=4, Hkv=2, D=8):
    q, k, v = (_rand((1, H, S, D), seed, t) for t, H in ((0, Hq), (1, Hkv), (2, Hkv)))
    rng = np.random.default_rng(seed)
    nt = (S + 127) // 128
    bm = (rng.random((Hq, nt, nt)) < 0.8).astype(np.uint8)
    keep = rng.random((1, S, S)) < 0.7
    bits = np.zeros((1, S, _keep_rows(S)), np.uint8)
    for jj in range(S):
        bits[:, :, jj // 8] |= (keep[:, :, jj].astype(np.uint8) << (jj % 8))
    return q, k, v, bm, keep, bits


def _combo_torch(qf, kf, vf, scale, causal, bm, keep, Z, s):
    Hq, S = qf.shape[1], qf.shape[2]
    em = _expand_block_mask(bm, Hq, S, False) & torch.from_numpy(keep).expand(Hq, S, S)
    if causal:
        em = em & torch.ones(S, S, dtype=torch.bool).tril()
    sc = torch.einsum("bhid,bhjd->bhij", qf, kf) * scale
    sc = sc.masked_fill(~em, float("-inf"))
    none = ~em.any(dim=-1)
    p = torch.softmax(sc.masked_fill(none[None, :, :, None], 0.0), dim=-1).masked_fill(~em, 0.0)
    return torch.einsum("bhij,bhjd->bhid", p * Z * s, vf), torch.logsumexp(sc, dim=-1), none


def pin_combo_library(attnx):
    """Block mask, keep bits and dropout together against the float64 formula in
    torch (masked softmax, rows without keys 0, weights times Z * 256/(256-p8) with
    Z from the test-side Philox4x32-10)."""
    q, k, v, bm, keep, bits = _combo_inputs(351)
    Hq, Hkv, S = 4, 2, 200
    p8, seed, offset = 60, 0xABC, 3
    Z = torch.from_numpy(np.stack([keep_table(h, S, p8, seed, offset) for h in range(Hq)])[None].astype(np.float64))
    sc32 = float(np.float32(0.3))
    qf = torch.from_numpy(f64(q))
    kf = torch.from_numpy(f64(k)).repeat_interleave(Hq // Hkv, 1)
    vf = torch.from_numpy(f64(v)).repeat_interleave(Hq // Hkv, 1)
    for causal in (True, False):
        O, L = attnx(q, k, v, 0.3, causal, block_mask=bm, keep_bits=bits, dropout=(p8, seed, offset))
        ref, lse, none = _combo_torch(qf, kf, vf, sc32, causal, bm, keep, Z, 256.0 / (256 - p8))
        np.testing.assert_allclose(O, ref.numpy(), rtol=0, atol=1e-12)
        live = ~none.numpy()
        np.testing.assert_allclose(L[0][live], lse.numpy()[0][live], rtol=0, atol=1e-12)
        assert np.all(np.isneginf(L[0][~live]))


def pin_combo_e4m3_masks(attnx):
    """E4M3 inputs with a block mask and keep bits against torch's float64 SDPA on
    the decoded values (torch's own float8_e4m3fn conversion) with the same mask."""
    from causal_scaled_dot_gb300.inputs import float32_to_e4m3_codes
    q, k, v, bm, keep, bits = _combo_inputs(361)
    Hq, Hkv, S = 4, 2, 200
    codes = [float32_to_e4m3_codes(f64(x).astype(np.float32)) for x in (q, k, v)]
    ds = (0.5, 2.0, 0.25)
    dec = [torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64) * d for c, d in zip(codes, ds)]
    qf, kf, vf = dec[0], dec[1].repeat_interleave(Hq // Hkv, 1), dec[2].repeat_interleave(Hq // Hkv, 1)
    for causal in (True, False):
        O, L = attnx(*codes, 0.3, causal, descales=ds, block_mask=bm, keep_bits=bits)
        ref, lse, none = _combo_torch(qf, kf, vf, float(np.float32(0.3)), causal, bm, keep, 1.0, 1.0)
        np.testing.assert_allclose(O, ref.numpy(), rtol=0, atol=1e-12)
        live = ~none.numpy()
        np.testing.assert_allclose(L[0][live], lse.numpy()[0][live], rtol=0, atol=1e-12)


COMBO_PINS = [pin_combo_library, pin_combo_e4m3_masks]


def pin_bwd_combo_autograd(bwdx):
    """Gradients with a block mask, keep bits and dropout together against torch's
    float64 autograd of the same formula."""
    q, k, v, bm, keep, bits = _combo_inputs(371)
    Hq, Hkv, S, D = 4, 2, 200, 8
    dout = _rand((1, Hq, S, D), 371, 3)
    G = Hq // Hkv
    p8, seed, offset = 25, 0x77, 1
    Z = torch.from_numpy(np.stack([keep_table(h, S, p8, seed, offset) for h in range(Hq)])[None].astype(np.float64))
    for causal in (True, False):
        dq, dk, dv, _ = bwdx(q, k, v, dout, 0.4, causal, bm, bits, (p8, seed, offset))
        tq, tk, tv = (torch.from_numpy(f64(x)).requires_grad_() for x in (q, k, v))
        o, _, _ = _combo_torch(tq, tk.repeat_interleave(G, 1), tv.repeat_interleave(G, 1),
                               float(np.float32(0.4)), causal, bm, keep, Z, 256.0 / (256 - p8))
        o.backward(torch.from_numpy(f64(dout)))
        for name, a, t in (("dQ", dq, tq), ("dK", dk, tk), ("dV", dv, tv)):
            ref = t.grad.numpy()
            assert np.max(np.abs(a - ref)) <= 1e-12 * max(1.0, float(np.max(np.abs(ref)))), name


BWD_COMBO_PINS = [pin_bwd_combo_autograd]
