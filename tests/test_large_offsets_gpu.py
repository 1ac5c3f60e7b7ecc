"""Large tensors: 131072 heads of 128 rows x 128 (2^31 elements, 4 GiB per bf16
tensor), so that row and head offsets pass 2^31 bytes and elements.  Inputs
come from torch's seeded device generator (the host generator would take
minutes at this size); the heads checked -- the first, the last and ones just
past the 2^31-byte boundary -- are copied to the host and compared with the
oracle on that head alone."""
import math

import numpy as np
import pytest

import oracle
from tests.gpu_util import bits_of, compare, compare_grad

pytestmark = pytest.mark.gpu

B, H, S, D = 1024, 128, 128, 128
HEADS = [0, 1, (1 << 30) // (S * D) - 1, (1 << 30) // (S * D), (1 << 30) // (S * D) + 7,
         B * H - 2, B * H - 1]  # head ids; 2^30 elements = 2^31 bytes


@pytest.fixture(scope="module")
def big():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    free, _ = torch.cuda.mem_get_info()
    if free < 48 * (1 << 30):
        pytest.skip("needs about 48 GiB of free device memory")
    g = torch.Generator(device="cuda").manual_seed(20261202)
    mk = lambda: torch.randn((B, H, S, D), generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)  # noqa: E731
    q = mk()
    k = mk()
    v = mk()
    yield q, k, v
    del q, k, v
    torch.cuda.empty_cache()


def _head(t, h):
    return bits_of(t.view(B * H, S, D)[h]).reshape(1, 1, S, D)


def test_forward_large_offsets(big):
    import torch
    from causal_scaled_dot_gb300 import native
    q, k, v = big
    out = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    native.attn_fwd(q, k, v, out, lse, B, H, H, S, D, D ** -0.5, True)
    native.attn_sync_status()
    for h in HEADS:
        o_ref, l_ref = oracle.attention(_head(q, h), _head(k, h), _head(v, h), D ** -0.5, True)
        o = out.view(B * H, S, D)[h].double().cpu().numpy().reshape(o_ref.shape)
        l = lse.view(B * H, S)[h].double().cpu().numpy().reshape(l_ref.shape)
        compare(o, o_ref, l, l_ref, f"head {h}")


def test_backward_and_projection_large_offsets(big):
    import torch
    from causal_scaled_dot_gb300 import native
    q, k, v = big
    out = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    native.attn_fwd(q, k, v, out, lse, B, H, H, S, D, D ** -0.5, True)
    g = torch.Generator(device="cuda").manual_seed(7)
    do = torch.randn(out.shape, generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    delta = torch.empty_like(lse)
    native.attn_bwd(q, k, v, out, do, lse, delta, dq, dk, dv, B, H, H, S, D, D ** -0.5, True)
    native.attn_sync_status()
    for h in HEADS:
        rq, rk, rv, _ = oracle.attention_bwd(_head(q, h), _head(k, h), _head(v, h), _head(do, h),
                                             D ** -0.5, True)
        for name, got, ref in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
            gh = got.view(B * H, S, D)[h].double().cpu().numpy().reshape(ref.shape)
            compare_grad(gh, ref, f"head {h} {name}")
    del dq, dk, dv, do
    # The projection of the same output: E = 256 features over K = H*D = 16384.
    E = 256
    w_bits = (torch.randn((E, H * D), generator=g, device="cuda") * (H * D) ** -0.5).to(torch.bfloat16)
    y = torch.empty((B, S, E), dtype=torch.bfloat16, device="cuda")
    native.attn_out_proj(out, w_bits, None, y, B, H, S, D, E)
    native.attn_sync_status()
    wb = bits_of(w_bits)
    for b in (0, B // 2, B - 1):
        ob = bits_of(out[b]).reshape(1, H, S, D)
        ref = oracle.out_proj(ob, wb)
        got = y[b].double().cpu().numpy().reshape(ref.shape)
        assert float(np.abs(got - ref).max()) <= 2.0 ** -8 * float(np.abs(ref).max()), f"batch {b}"
