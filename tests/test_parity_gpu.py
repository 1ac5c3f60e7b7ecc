"""GPU parity: libattn (through its C ABI) against the fp64 CPU oracle on the
same seeded bf16 inputs.  Tolerances: bf16 O max abs <= 2e-2 and relative L2
<= 5e-3, fp32 LSE max abs <= 1e-3."""
import math

import numpy as np
import pytest

import oracle
from causal_scaled_dot_gb300.inputs import (bf16_bits_to_float32, float32_to_bf16_bits,
                                            gaussian_bf16, qkv_bf16)
from causal_scaled_dot_gb300.workloads import SMALL, WORKLOADS
from tests.gpu_util import compare, run_gpu, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True, params=["ws", "simple"])
def kernel(request):
    """Every test runs on both kernels: the warp-specialised persistent one
    (the default) and the one-tile-per-CTA one (ATTN_FWD_KERNEL=simple)."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os
    from causal_scaled_dot_gb300 import native
    native.load()
    old = os.environ.get("ATTN_FWD_KERNEL")
    os.environ["ATTN_FWD_KERNEL"] = request.param
    yield request.param
    if old is None:
        os.environ.pop("ATTN_FWD_KERNEL", None)
    else:
        os.environ["ATTN_FWD_KERNEL"] = old


def _check(B, Hq, Hkv, S, D, causal, seed, sigma=1.0, scale=None):
    q, k, v = qkv_bf16(B, Hq, Hkv, S, D, seed=seed, sigma=sigma)
    scale = scale or 1.0 / math.sqrt(D)
    o, l, _ = run_gpu(q, k, v, scale, causal)
    o_ref, l_ref = oracle.attention(q, k, v, scale, causal)
    return compare(o, o_ref, l, l_ref, f"B{B} Hq{Hq} Hkv{Hkv} S{S} D{D} causal={causal}")


def test_small_workload_all_rows():
    w = SMALL
    _check(w.B, w.Hq, w.Hkv, w.S, w.D, True, w.seed, w.sigma)


@pytest.mark.parametrize("S", [1, 2, 63, 127, 128, 129, 255, 300, 1000])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_sequence_lengths(S, D, causal):
    _check(1, 2, 1, S, D, causal, seed=100 + S)


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 2), (8, 2), (8, 1), (32, 1)])
@pytest.mark.parametrize("B", [1, 3])
def test_head_groups_and_batches(B, Hq, Hkv):
    _check(B, Hq, Hkv, 200, 128, True, seed=200 + Hq * 10 + Hkv + B)


def test_d64_multi_tile_gqa():
    _check(2, 8, 2, 700, 64, True, seed=301)


@pytest.mark.parametrize("B,H,S,D", [(8, 64, 256, 128), (3, 100, 1024, 128), (5, 40, 640, 64),
                                     (1, 1, 4096, 128), (2, 3, 2200, 64)])
def test_many_units_per_cta(B, H, S, D):
    """More units than SMs, so every CTA of the persistent kernel runs several
    units and its K/V ring wraps many times; sampled rows against the oracle."""
    q, k, v = qkv_bf16(B, H, H, S, D, seed=B * 1000 + S)
    o, l, _ = run_gpu(q, k, v, 1 / math.sqrt(D), True)
    rows = sample_rows(B, H, S, n_random=512, seed=S)
    o_ref, l_ref = oracle.attention(q, k, v, 1 / math.sqrt(D), True, rows=rows)
    compare(o.reshape(-1, D)[rows], o_ref, l.reshape(-1)[rows], l_ref, f"B{B} H{H} S{S} D{D}")
    assert np.all(np.isfinite(o))


@pytest.mark.parametrize("w", WORKLOADS[1:], ids=lambda w: w.name)
def test_full_size_workloads_sampled_rows(w):
    """Each workload at full size; the oracle recomputes a sample of rows."""
    q, k, v = qkv_bf16(w.B, w.Hq, w.Hkv, w.S, w.D, seed=w.seed, sigma=w.sigma)
    o, l, _ = run_gpu(q, k, v, w.scale, w.causal)
    rows = sample_rows(w.B, w.Hq, w.S, n_random=384, seed=w.seed)
    o_ref, l_ref = oracle.attention(q, k, v, w.scale, w.causal, rows=rows)
    stats = compare(o.reshape(-1, w.D)[rows], o_ref, l.reshape(-1)[rows], l_ref, w.name)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l)), "some output row was not written"
    print(w.name, stats)


def test_causal_row0_is_bit_exact_v0():
    """Row 0 attends to key 0 alone, so O_0 = V_0 exactly in bf16."""
    q, k, v = qkv_bf16(2, 4, 2, 300, 128, seed=401)
    _, l, obits = run_gpu(q, k, v, 1 / math.sqrt(128), True)
    assert np.array_equal(obits[:, :, 0, :], np.repeat(v, 2, axis=1)[:, :, 0, :])
    qf = bf16_bits_to_float32(q).astype(np.float64)
    kf = np.repeat(bf16_bits_to_float32(k).astype(np.float64), 2, axis=1)
    l0 = np.einsum("bhd,bhd->bh", qf[:, :, 0], kf[:, :, 0]) * float(np.float32(1 / math.sqrt(128)))
    np.testing.assert_allclose(l[:, :, 0], l0, rtol=0, atol=1e-4)


def test_q_zero_gives_prefix_means():
    B, Hq, Hkv, S, D = 1, 2, 2, 333, 128
    q = np.zeros((B, Hq, S, D), np.uint16)
    k = gaussian_bf16((B, Hkv, S, D), 501, 1)
    v = gaussian_bf16((B, Hkv, S, D), 501, 2)
    o, l, _ = run_gpu(q, k, v, 0.125, True)
    vf = bf16_bits_to_float32(v).astype(np.float64)
    counts = np.arange(1, S + 1)[None, None, :, None]
    compare(o, np.cumsum(vf, axis=2) / counts, l, np.broadcast_to(np.log(counts[..., 0]), l.shape),
            "Q=0")


def test_causality_is_bitwise():
    """Changing keys/values after position i leaves rows <= i bit-identical."""
    B, H, S, D = 1, 2, 384, 128
    q, k, v = qkv_bf16(B, H, H, S, D, seed=601)
    _, l1, o1 = run_gpu(q, k, v, 0.09, True)
    cut = 150
    k2, v2 = k.copy(), v.copy()
    k2[:, :, cut + 1:] = gaussian_bf16((B, H, S - cut - 1, D), 602, 1)
    v2[:, :, cut + 1:] = gaussian_bf16((B, H, S - cut - 1, D), 602, 2)
    _, l2, o2 = run_gpu(q, k2, v2, 0.09, True)
    assert np.array_equal(o1[:, :, :cut + 1], o2[:, :, :cut + 1])
    assert np.array_equal(l1[:, :, :cut + 1], l2[:, :, :cut + 1])
    assert not np.array_equal(o1[:, :, cut + 1:], o2[:, :, cut + 1:])


def test_repeated_calls_are_bitwise_equal():
    q, k, v = qkv_bf16(2, 8, 4, 1000, 128, seed=701)
    _, l1, o1 = run_gpu(q, k, v, 0.088, True)
    _, l2, o2 = run_gpu(q, k, v, 0.088, True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_large_magnitude_scores():
    """Q x 8 pushes the scores far from 0; the running max keeps exp2 in range."""
    q, k, v = qkv_bf16(1, 4, 4, 520, 128, seed=801)
    q = float32_to_bf16_bits(bf16_bits_to_float32(q) * np.float32(8.0))
    o, l, _ = run_gpu(q, k, v, 1 / math.sqrt(128), True)
    o_ref, l_ref = oracle.attention(q, k, v, 1 / math.sqrt(128), True)
    compare(o, o_ref, l, l_ref, "Qx8")


def test_lse_null_is_allowed():
    q, k, v = qkv_bf16(1, 2, 2, 130, 64, seed=901)
    o, _, _ = run_gpu(q, k, v, 0.125, True, with_lse=False)
    o_ref, _ = oracle.attention(q, k, v, 0.125, True)
    compare(o, o_ref, None, None, "lse=NULL")


def test_nothing_written_outside_the_outputs():
    """Guard regions around out and lse stay untouched (ragged S, D = 64 and 128)."""
    import torch
    from causal_scaled_dot_gb300 import native
    from tests.gpu_util import to_device
    for D in (64, 128):
        B, H, S = 1, 3, 200
        q, k, v = qkv_bf16(B, H, H, S, D, seed=1001 + D)
        qd, kd, vd = to_device(q), to_device(k), to_device(v)
        n = B * H * S * D
        guard = 4096
        obuf = torch.full((n + 2 * guard,), 7.0, dtype=torch.bfloat16, device="cuda")
        lbuf = torch.full((B * H * S + 2 * guard,), 7.0, dtype=torch.float32, device="cuda")
        out = obuf[guard:guard + n]
        lse = lbuf[guard:guard + B * H * S]
        native.attn_fwd(qd, kd, vd, out, lse, B, H, H, S, D, 1 / math.sqrt(D), True)
        native.attn_sync_status()
        assert torch.all(obuf[:guard] == 7.0) and torch.all(obuf[guard + n:] == 7.0)
        assert torch.all(lbuf[:guard] == 7.0) and torch.all(lbuf[guard + B * H * S:] == 7.0)
        assert torch.all(torch.isfinite(out.float()))


def test_bounded_wait_reports_timeout_and_device_stays_usable():
    """A wait on a barrier nobody arrives at gives up after its limit, the kernel
    returns, the status word reports the timeout, and later calls still work."""
    from causal_scaled_dot_gb300 import native
    assert native.attn_selftest_wait_timeout(2000) == native.ATTN_OK
    assert native.attn_sync_status(check=False) == native.ATTN_ERR_TIMEOUT
    assert native.attn_sync_status(check=False) == native.ATTN_OK  # cleared by the read
    test_small_workload_all_rows()


def test_binding_rejects_non_contiguous_tensors():
    import torch
    from causal_scaled_dot_gb300 import native
    q = torch.zeros((1, 2, 128, 64), dtype=torch.bfloat16, device="cuda")
    qt = q.transpose(2, 3)
    with pytest.raises(ValueError):
        native.attn_fwd(qt, q, q, torch.empty_like(q), None, 1, 2, 2, 128, 64, 0.125, True)
