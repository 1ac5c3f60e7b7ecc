"""GPU parity of the output projection (attn_out_proj) against the oracle's
float64 definition.  Tolerance: one bf16 rounding of each output (<= 2^-9
relative) and fp32 accumulation (negligible at these K), with a factor 2:
max abs <= 2^-8 * max|Y|, relative L2 <= 2^-8."""
import numpy as np
import pytest

import oracle
from causal_scaled_dot_gb300.inputs import gaussian_bf16
from causal_scaled_dot_gb300.workloads import WORKLOADS
from tests.gpu_util import bits_of, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_proj(o_bits, w_bits, bias):
    import torch
    from causal_scaled_dot_gb300 import native
    B, H, S, D = o_bits.shape
    E = w_bits.shape[0]
    o, w = to_device(o_bits), to_device(w_bits)
    b = torch.from_numpy(np.asarray(bias, dtype=np.float32)).cuda() if bias is not None else None
    y = torch.full((B, S, E), float("nan"), dtype=torch.bfloat16, device="cuda")
    native.attn_out_proj(o, w, b, y, B, H, S, D, E)
    native.attn_sync_status(None)
    return y.double().cpu().numpy()


def _check(B, H, S, D, E, seed, with_bias=True):
    o = gaussian_bf16((B, H, S, D), seed, 0)
    w = gaussian_bf16((E, H * D), seed, 1, sigma=1.0 / np.sqrt(H * D))
    bias = np.random.default_rng(seed).standard_normal(E).astype(np.float32) if with_bias else None
    y = run_proj(o, w, bias)
    ref = oracle.out_proj(o, w, bias)
    assert np.all(np.isfinite(y)), "unwritten outputs"
    err = np.abs(y - ref)
    max_abs, scale = float(err.max()), float(np.abs(ref).max())
    rel_l2 = float(np.linalg.norm(y - ref) / np.linalg.norm(ref))
    label = f"proj B{B} H{H} S{S} D{D} E{E}"
    assert max_abs <= 2.0 ** -8 * scale, f"{label}: max abs {max_abs:.3e} > {2.0 ** -8 * scale:.3e}"
    assert rel_l2 <= 2.0 ** -8, f"{label}: rel L2 {rel_l2:.3e}"
    return {"max_abs": max_abs, "rel_l2": rel_l2}


@pytest.mark.parametrize("S", [1, 127, 128, 129, 300])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("E", [8, 248, 256, 264, 1000])
def test_proj_shapes(S, D, E):
    print(_check(2, 3, S, D, E, seed=4100 + S + D + E))


def test_proj_without_bias():
    print(_check(1, 4, 200, 128, 512, seed=4200, with_bias=False))


def test_proj_many_tiles_per_cta():
    print(_check(3, 8, 1000, 128, 1536, seed=4300))


@pytest.mark.parametrize("w", WORKLOADS[1:4], ids=lambda w: w.name)
def test_proj_full_size_workloads(w):
    """The projection of each attention workload's output: E = Hq * D."""
    print(w.name, _check(w.B, w.Hq, w.S, w.D, w.Hq * w.D, seed=w.seed))


def test_proj_reads_attention_output_in_place():
    """attn_fwd, then attn_out_proj on the same buffer, equals the oracle
    projection of the GPU's own attention output."""
    import torch
    from causal_scaled_dot_gb300 import native
    from causal_scaled_dot_gb300.inputs import qkv_bf16
    B, H, S, D, E = 2, 4, 384, 128, 512
    q, k, v = qkv_bf16(B, H, H, S, D, seed=4400)
    qd, kd, vd = to_device(q), to_device(k), to_device(v)
    out = torch.empty_like(qd)
    native.attn_fwd(qd, kd, vd, out, None, B, H, H, S, D, D ** -0.5, True)
    w = gaussian_bf16((E, H * D), 4400, 5, sigma=1.0 / np.sqrt(H * D))
    y = torch.empty((B, S, E), dtype=torch.bfloat16, device="cuda")
    native.attn_out_proj(out, to_device(w), None, y, B, H, S, D, E)
    native.attn_sync_status(None)
    ref = oracle.out_proj(bits_of(out), w, None)
    got = y.double().cpu().numpy()
    assert float(np.abs(got - ref).max()) <= 2.0 ** -8 * float(np.abs(ref).max())
