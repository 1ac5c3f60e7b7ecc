"""Helpers for the GPU parity tests: move seeded bf16 bits to the device, run
libattn through its C ABI, and compare with the fp64 oracle."""
from __future__ import annotations

import math

import numpy as np

# Tolerances on bf16 O against the fp64 oracle, and on fp32 LSE.
TOL_O_MAX_ABS = 2e-2
TOL_O_REL_L2 = 5e-3
TOL_LSE_MAX_ABS = 1e-3


def to_device(bits: np.ndarray):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy())
    return t.view(torch.bfloat16).cuda()


def bits_of(t) -> np.ndarray:
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def run_gpu(q_bits, k_bits, v_bits, scale, causal, with_lse=True, stream=None):
    """attn_fwd through the C ABI; returns (O float64, LSE float64 or None, O bf16 bits)."""
    import torch
    from causal_scaled_dot_gb300 import native
    B, Hq, S, D = q_bits.shape
    Hkv = k_bits.shape[1]
    q, k, v = to_device(q_bits), to_device(k_bits), to_device(v_bits)
    out = torch.full_like(q, float("nan"))  # unwritten rows would stay NaN
    lse = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    native.attn_fwd(q, k, v, out, lse, B, Hq, Hkv, S, D, scale, causal, stream=stream)
    native.attn_sync_status(stream)
    o = out.double().cpu().numpy()
    l = lse.double().cpu().numpy() if with_lse else None
    return o, l, bits_of(out)


def compare(o_gpu, o_ref, l_gpu, l_ref, label="", abs_scale=1.0):
    """Assert the parity bar; returns the error figures.  ``abs_scale`` widens
    the max-abs bound for outputs that are a known factor larger (dropout's
    256 / (256 - p8)); the relative L2 bound does not change."""
    assert np.all(np.isfinite(o_gpu)), f"{label}: non-finite output (unwritten rows?)"
    diff = o_gpu - o_ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    ref_norm = float(np.linalg.norm(o_ref))
    rel_l2 = float(np.linalg.norm(diff) / ref_norm) if ref_norm > 0 else float(np.linalg.norm(diff))
    stats = {"max_abs": max_abs, "rel_l2": rel_l2}
    assert max_abs <= TOL_O_MAX_ABS * abs_scale, \
        f"{label}: O max abs error {max_abs:.3e} > {TOL_O_MAX_ABS * abs_scale}"
    assert rel_l2 <= TOL_O_REL_L2, f"{label}: O rel L2 error {rel_l2:.3e} > {TOL_O_REL_L2}"
    if l_gpu is not None:
        assert np.all(np.isfinite(l_gpu)), f"{label}: non-finite LSE"
        lse_err = float(np.max(np.abs(l_gpu - l_ref))) if l_gpu.size else 0.0
        stats["lse_max_abs"] = lse_err
        assert lse_err <= TOL_LSE_MAX_ABS, f"{label}: LSE max abs error {lse_err:.3e} > {TOL_LSE_MAX_ABS}"
    return stats


def sample_rows(B, Hq, S, n_random=256, seed=0):
    """Flat row ids covering both ends of the sequence, tile edges and random rows."""
    rng = np.random.default_rng(seed)
    heads = {(0, 0), (B - 1, Hq - 1), (0, Hq - 1), (B - 1, 0)}
    for _ in range(4):
        heads.add((int(rng.integers(B)), int(rng.integers(Hq))))
    positions = {0, 1, 2, 127, 128, 129, 255, 256, S // 2, S - 129, S - 128, S - 127, S - 2, S - 1}
    rows = {(b * Hq + h) * S + i for (b, h) in heads for i in positions if 0 <= i < S}
    rows |= set(int(x) for x in rng.integers(0, B * Hq * S, size=n_random))
    return np.array(sorted(rows), dtype=np.int64)


def run_gpu_fp8(q_codes, k_codes, v_codes, descales, scale, causal, with_lse=True, stream=None):
    """attn_fwd_fp8 through the C ABI on E4M3 codes; returns (O float64, LSE float64 or None)."""
    import torch
    from causal_scaled_dot_gb300 import native
    B, Hq, S, D = q_codes.shape
    Hkv = k_codes.shape[1]
    dev = lambda c: torch.from_numpy(np.ascontiguousarray(c)).cuda()  # noqa: E731
    q, k, v = dev(q_codes), dev(k_codes), dev(v_codes)
    out = torch.full((B, Hq, S, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    native.attn_fwd_fp8(q, k, v, *descales, out, lse, B, Hq, Hkv, S, D, scale, causal, stream=stream)
    native.attn_sync_status(stream)
    return out.double().cpu().numpy(), (lse.double().cpu().numpy() if with_lse else None)


def fp8_tolerances(v_values, o_ref):
    """Bounds for FP8 inputs.  The probabilities that multiply V are rounded to
    E4M3 (3 mantissa bits, round to nearest: relative error <= 2^-4 each), so a
    row of O moves by at most 2^-4 * max|V| (the weights sum to 1); bf16 output
    rounding adds 2^-9 * |O|, taken twice.  The relative L2 bound is the
    per-weight bound 2^-4.  LSE uses the unrounded fp32 probabilities: 1e-3 as
    for bf16 inputs."""
    max_abs = 2.0 ** -4 * float(np.max(np.abs(v_values))) + 2.0 ** -8 * float(np.max(np.abs(o_ref)))
    return max_abs, 2.0 ** -4, TOL_LSE_MAX_ABS


def fp8_rounding_model(q_codes, k_codes, v_codes, descales, scale, causal, rows=None):
    """Relative L2 error of O that rounding the probabilities to E4M3 gives on
    these inputs, in a model of the kernel: the exact scores t_ij (log2 units),
    weights 2^(t_ij - M_i) with M_i the row maximum, each rounded to E4M3 with
    round-to-nearest-even (torch's float8_e4m3fn conversion), and
    O_i = sum_j round(w_ij) v_j / sum_j w_ij (the row sum stays unrounded, as in
    the kernel) against the same sum with unrounded weights; over the given
    flat rows (b*Hq + h)*S + i, or all rows.

    The kernel's reference maximum lies 0 to 8 binades below M_i (it is the
    first key tile's maximum unless a later tile exceeds it by more than 8), so
    its probabilities are the model's times one factor per row: relative
    rounding errors of normal E4M3 numbers have the same distribution, and
    fewer probabilities fall below the normal range than in the model."""
    import torch
    import oracle
    q = oracle.e4m3_decode(q_codes) * descales[0]
    k = oracle.e4m3_decode(k_codes) * descales[1]
    v = oracle.e4m3_decode(v_codes) * descales[2]
    B, Hq, S, D = q.shape
    G = Hq // k.shape[1]
    rows = np.arange(B * Hq * S) if rows is None else np.asarray(rows)
    num = den = 0.0
    for bh in np.unique(rows // S):
        b, h = divmod(int(bh), Hq)
        ii = rows[rows // S == bh] % S
        t = (q[b, h, ii] @ k[b, h // G].T) * (float(np.float32(scale)) / math.log(2.0))
        if causal:
            t = np.where(np.arange(S)[None, :] > ii[:, None], -np.inf, t)
        w = np.exp2(t - t.max(axis=1, keepdims=True))
        wq = torch.from_numpy(w).to(torch.float8_e4m3fn).double().numpy()
        l = w.sum(axis=1, keepdims=True)
        o = (w @ v[b, h // G]) / l
        oq = (wq @ v[b, h // G]) / l
        num += float(((oq - o) ** 2).sum())
        den += float((o ** 2).sum())
    return math.sqrt(num / den) if den > 0 else 0.0


def compare_fp8(o_gpu, o_ref, l_gpu, l_ref, v_values, label="", model_rel=None):
    """As ``fp8_tolerances``; with ``model_rel`` (``fp8_rounding_model`` on the
    same inputs and rows) the relative L2 bound tightens to twice the model's
    error plus 2^-8 (the bf16 output rounding, 2^-9, taken twice), never above
    the worst-case 2^-4."""
    tol_abs, tol_rel, tol_lse = fp8_tolerances(v_values, o_ref)
    if model_rel is not None:
        tol_rel = min(tol_rel, 2.0 * model_rel + 2.0 ** -8)
    assert np.all(np.isfinite(o_gpu)), f"{label}: non-finite output (unwritten rows?)"
    diff = o_gpu - o_ref
    max_abs = float(np.max(np.abs(diff)))
    rel_l2 = float(np.linalg.norm(diff) / np.linalg.norm(o_ref))
    stats = {"max_abs": max_abs, "rel_l2": rel_l2, "tol_abs": tol_abs, "tol_rel": tol_rel}
    assert max_abs <= tol_abs, f"{label}: O max abs error {max_abs:.3e} > {tol_abs:.3e}"
    assert rel_l2 <= tol_rel, f"{label}: O rel L2 error {rel_l2:.3e} > {tol_rel:.3e}"
    if l_gpu is not None:
        lse_err = float(np.max(np.abs(l_gpu - l_ref)))
        stats["lse_max_abs"] = lse_err
        assert lse_err <= tol_lse, f"{label}: LSE max abs error {lse_err:.3e} > {tol_lse}"
    return stats


def run_gpu_masked(q_bits, k_bits, v_bits, scale, causal, block_mask, stream=None):
    """attn_fwd_block_masked through the C ABI; returns (O float64, LSE float64)."""
    import torch
    from causal_scaled_dot_gb300 import native
    B, Hq, S, D = q_bits.shape
    Hkv = k_bits.shape[1]
    q, k, v = to_device(q_bits), to_device(k_bits), to_device(v_bits)
    m = torch.from_numpy(np.ascontiguousarray(block_mask, dtype=np.uint8)).cuda()
    out = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device="cuda")
    native.attn_fwd_block_masked(q, k, v, out, lse, B, Hq, Hkv, S, D, scale, causal, m,
                                 block_mask.shape[0], stream=stream)
    native.attn_sync_status(stream)
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def compare_masked(o_gpu, o_ref, l_gpu, l_ref, label="", abs_scale=1.0):
    """The bf16 parity bar on rows that see at least one key; rows that see none
    must hold exactly O = 0 and LSE = -inf on both sides."""
    D = o_ref.shape[-1]
    o_gpu, o_ref = o_gpu.reshape(-1, D), o_ref.reshape(-1, D)
    l_gpu, l_ref = l_gpu.reshape(-1), l_ref.reshape(-1)
    empty = np.isneginf(l_ref)
    assert np.all(np.isneginf(l_gpu[empty])), f"{label}: LSE of rows without keys is not -inf"
    assert np.all(o_gpu[empty] == 0.0), f"{label}: O of rows without keys is not 0"
    assert np.all(o_ref[empty] == 0.0)
    live = ~empty
    stats = {"empty_rows": int(empty.sum())}
    if live.any():
        stats.update(compare(o_gpu[live], o_ref[live], l_gpu[live], l_ref[live], label, abs_scale))
    return stats


# Backward: tolerances on bf16 dQ, dK, dV against the fp64 oracle.  A term of
# each product carries at most two bf16 roundings (P or dS, then the output),
# and delta comes from the bf16 forward output, each <= 2^-9 relative; under
# independent rounding errors that is about 3 * 2^-9 = 0.006 relative L2, so
# 1e-2 is the bound; the largest element error stays within 2 % of the
# tensor's largest magnitude.
TOL_GRAD_REL_L2 = 1e-2
TOL_GRAD_MAX_REL = 2e-2


def run_gpu_bwd(q_bits, k_bits, v_bits, do_bits, scale, causal, stream=None):
    """attn_fwd then attn_bwd through the C ABI on the same device buffers.
    Returns float64 (O, LSE, dQ, dK, dV, delta)."""
    import torch
    from causal_scaled_dot_gb300 import native
    B, Hq, S, D = q_bits.shape
    Hkv = k_bits.shape[1]
    q, k, v, do = to_device(q_bits), to_device(k_bits), to_device(v_bits), to_device(do_bits)
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    native.attn_fwd(q, k, v, out, lse, B, Hq, Hkv, S, D, scale, causal, stream=stream)
    dq = torch.full_like(q, float("nan"))
    dk = torch.full_like(k, float("nan"))
    dv = torch.full_like(v, float("nan"))
    delta = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device="cuda")
    native.attn_bwd(q, k, v, out, do, lse, delta, dq, dk, dv, B, Hq, Hkv, S, D, scale, causal,
                    stream=stream)
    native.attn_sync_status(stream)
    return tuple(t.double().cpu().numpy() for t in (out, lse, dq, dk, dv, delta))


def compare_grad(g, ref, label, abs_err: float = 0.0):
    """Relative L2 and largest error against the tensor's largest magnitude, with
    an absolute floor of 1e-3 per element: a gradient that is exactly 0 (causal
    row 0's dQ, a single key) is compared absolutely.  ``abs_err`` is a bound on
    an additive per-element error known from the arithmetic (it is taken off
    each element's error before the relative checks)."""
    assert np.all(np.isfinite(g)), f"{label}: non-finite values (unwritten rows?)"
    if ref.size == 0:
        return {}
    err = np.maximum(np.abs(g - ref) - abs_err, 0.0)
    floor = 1e-3
    rel_l2 = float(np.linalg.norm(err) / max(np.linalg.norm(ref), floor * math.sqrt(ref.size)))
    max_rel = float(np.max(err)) / max(float(np.max(np.abs(ref))), floor)
    assert rel_l2 <= TOL_GRAD_REL_L2, f"{label}: rel L2 {rel_l2:.3e} > {TOL_GRAD_REL_L2}"
    assert max_rel <= TOL_GRAD_MAX_REL, f"{label}: max abs / max|ref| {max_rel:.3e} > {TOL_GRAD_MAX_REL}"
    return {"rel_l2": rel_l2, "max_rel": max_rel}


def compare_delta(delta, delta_ref, o_ref, do, label):
    """delta_i = dO_i . O_i with O rounded to bf16: per row at most
    2^-8 * sum_d |dO_id O_id| apart (one bf16 rounding, margin 2), plus fp32 sums."""
    tol = 2.0 ** -8 * np.sum(np.abs(do * o_ref), axis=-1) + 1e-5
    err = np.abs(delta - delta_ref)
    assert np.all(err <= tol), f"{label}: delta error {float(np.max(err - tol)):.3e} over its bound"
    return float(np.max(err))


def run_gpu_dropout(q_bits, k_bits, v_bits, scale, causal, dropout_p, seed, offset, stream=None):
    """attn_fwd_dropout through the C ABI; returns (O float64, LSE float64)."""
    import torch
    from causal_scaled_dot_gb300 import native
    B, Hq, S, D = q_bits.shape
    Hkv = k_bits.shape[1]
    q, k, v = to_device(q_bits), to_device(k_bits), to_device(v_bits)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device="cuda")
    native.attn_fwd_dropout(q, k, v, out, lse, B, Hq, Hkv, S, D, scale, causal, dropout_p, seed,
                            offset, stream=stream)
    native.attn_sync_status(stream)
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def run_gpu_bwd_masked(q_bits, k_bits, v_bits, do_bits, scale, causal, block_mask, stream=None):
    """attn_fwd_block_masked then attn_bwd_block_masked on the same buffers.
    Returns float64 (O, LSE, dQ, dK, dV, delta)."""
    import torch
    from causal_scaled_dot_gb300 import native
    B, Hq, S, D = q_bits.shape
    Hkv = k_bits.shape[1]
    q, k, v, do = to_device(q_bits), to_device(k_bits), to_device(v_bits), to_device(do_bits)
    m = torch.from_numpy(np.ascontiguousarray(block_mask, dtype=np.uint8)).cuda()
    hm = block_mask.shape[0]
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    native.attn_fwd_block_masked(q, k, v, out, lse, B, Hq, Hkv, S, D, scale, causal, m, hm,
                                 stream=stream)
    dq = torch.full_like(q, float("nan"))
    dk = torch.full_like(k, float("nan"))
    dv = torch.full_like(v, float("nan"))
    delta = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device="cuda")
    native.attn_bwd_block_masked(q, k, v, out, do, lse, delta, dq, dk, dv, B, Hq, Hkv, S, D, scale,
                                 causal, m, hm, stream=stream)
    native.attn_sync_status(stream)
    return tuple(t.double().cpu().numpy() for t in (out, lse, dq, dk, dv, delta))


def run_gpu_elem_masked(q_bits, k_bits, v_bits, scale, causal, keep_bits, block_mask=None,
                        stream=None):
    """attn_fwd_elem_masked through the C ABI; returns (O float64, LSE float64)."""
    import torch
    from causal_scaled_dot_gb300 import native
    B, Hq, S, D = q_bits.shape
    Hkv = k_bits.shape[1]
    q, k, v = to_device(q_bits), to_device(k_bits), to_device(v_bits)
    kb = torch.from_numpy(np.ascontiguousarray(keep_bits, dtype=np.uint8)).cuda()
    bm = None if block_mask is None else torch.from_numpy(np.ascontiguousarray(block_mask, dtype=np.uint8)).cuda()
    out = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device="cuda")
    native.attn_fwd_elem_masked(q, k, v, out, lse, B, Hq, Hkv, S, D, scale, causal, kb,
                                keep_bits.shape[0], bm, 1 if block_mask is None else block_mask.shape[0],
                                stream=stream)
    native.attn_sync_status(stream)
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def run_gpu_bwd_elem_masked(q_bits, k_bits, v_bits, do_bits, scale, causal, keep_bits,
                            block_mask=None, stream=None):
    """attn_fwd_elem_masked then attn_bwd_elem_masked on the same buffers.
    Returns float64 (O, LSE, dQ, dK, dV, delta)."""
    import torch
    from causal_scaled_dot_gb300 import native
    B, Hq, S, D = q_bits.shape
    Hkv = k_bits.shape[1]
    q, k, v, do = to_device(q_bits), to_device(k_bits), to_device(v_bits), to_device(do_bits)
    kb = torch.from_numpy(np.ascontiguousarray(keep_bits, dtype=np.uint8)).cuda()
    bm = None if block_mask is None else torch.from_numpy(np.ascontiguousarray(block_mask, dtype=np.uint8)).cuda()
    hk, hm = keep_bits.shape[0], 1 if block_mask is None else block_mask.shape[0]
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    native.attn_fwd_elem_masked(q, k, v, out, lse, B, Hq, Hkv, S, D, scale, causal, kb, hk, bm, hm,
                                stream=stream)
    dq = torch.full_like(q, float("nan"))
    dk = torch.full_like(k, float("nan"))
    dv = torch.full_like(v, float("nan"))
    delta = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device="cuda")
    native.attn_bwd_elem_masked(q, k, v, out, do, lse, delta, dq, dk, dv, B, Hq, Hkv, S, D, scale,
                                causal, kb, hk, bm, hm, stream=stream)
    native.attn_sync_status(stream)
    return tuple(t.double().cpu().numpy() for t in (out, lse, dq, dk, dv, delta))


def run_gpu_bwd_dropout(q_bits, k_bits, v_bits, do_bits, scale, causal, dropout_p, seed, offset,
                        stream=None):
    """attn_fwd_dropout then attn_bwd_dropout on the same buffers.
    Returns float64 (O, LSE, dQ, dK, dV, delta)."""
    import torch
    from causal_scaled_dot_gb300 import native
    B, Hq, S, D = q_bits.shape
    Hkv = k_bits.shape[1]
    q, k, v, do = to_device(q_bits), to_device(k_bits), to_device(v_bits), to_device(do_bits)
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    native.attn_fwd_dropout(q, k, v, out, lse, B, Hq, Hkv, S, D, scale, causal, dropout_p, seed, offset,
                            stream=stream)
    dq = torch.full_like(q, float("nan"))
    dk = torch.full_like(k, float("nan"))
    dv = torch.full_like(v, float("nan"))
    delta = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device="cuda")
    native.attn_bwd_dropout(q, k, v, out, do, lse, delta, dq, dk, dv, B, Hq, Hkv, S, D, scale, causal,
                            dropout_p, seed, offset, stream=stream)
    native.attn_sync_status(stream)
    return tuple(t.double().cpu().numpy() for t in (out, lse, dq, dk, dv, delta))
