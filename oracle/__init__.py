"""fp64 CPU oracle for causal scaled dot-product attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg import this package (``__graft_entry__.build()`` compiles it without using
it).  The CUDA library never links, loads or calls it, and it imports nothing
from the CUDA library's package.

The arithmetic lives in ``attn_oracle.c`` (plain C, double precision, one query
row at a time, the five steps of the naive causal attention in the order the
"Profiling in PyTorch (Part 3)" retelling lists them in its section "Naive
Attention").  This module only builds that file with gcc and marshals numpy
arrays into it.

It also holds the gradients of the same function (``attention_bwd``: dQ, dK,
dV and the row term delta for an upstream gradient dO), written out as the
plain derivative in double precision.

Parity status: pinned.  ``tests/test_oracle_pins.py`` checks it against
library float64 routines, closed forms and invariants; ``tests/test_oracle_mutants.py``
plants mistakes into copies of the C source and checks that a pin catches each.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "attn_oracle.c")
BUILD_DIR = os.path.join(_HERE, "_build")
LIBRARY = os.path.join(BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_lib_cache: dict[str, ctypes.CDLL] = {}


def compile_oracle(source: str = SOURCE, output: str = LIBRARY) -> str:
    """Compile ``source`` into a shared library at ``output`` with gcc.

    Plain ``-O2`` without fast-math or machine-specific flags, so the same
    results come out on x86_64 and aarch64 hosts.
    """
    os.makedirs(os.path.dirname(output), exist_ok=True)
    tmp = output + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, source, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, output)
    return output


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    vp, ci, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f = lib.oracle_attn_rows
    f.restype = ci
    f.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, vp, ctypes.c_int64, vp, vp, ci]
    f = lib.oracle_attn_rows_e4m3
    f.restype = ci
    f.argtypes = [vp, vp, vp, cf, cf, cf, ci, ci, ci, ci, ci, cf, ci, vp, ctypes.c_int64, vp, vp,
                  ci]
    f = lib.oracle_attn_rows_masked
    f.restype = ci
    f.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, vp, ci, vp, ctypes.c_int64, vp, vp, ci]
    f = lib.oracle_e4m3_decode
    f.restype = None
    f.argtypes = [vp, ctypes.c_int64, vp]
    f = lib.oracle_attn_rows_f64
    f.restype = ci
    f.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, vp, ctypes.c_int64, vp, vp, ci]
    f = lib.oracle_attn_bwd_masked
    f.restype = ci
    f.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, vp, ci, vp, ctypes.c_int64, vp, vp,
                  vp, vp, ci]
    f = lib.oracle_attn_rows_dropout
    f.restype = ci
    f.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, ci, ctypes.c_uint64, ctypes.c_uint64, vp,
                  ctypes.c_int64, vp, vp, ci]
    f = lib.oracle_philox4x32
    f.restype = None
    f.argtypes = [vp, vp, vp]
    f = lib.oracle_attn_bwd
    f.restype = ci
    f.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, vp, ctypes.c_int64, vp, vp, vp,
                  vp, ci]
    f = lib.oracle_attn_rows_keep
    f.restype = ci
    f.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, vp, ci, vp, ci, vp, ctypes.c_int64, vp, vp,
                  ci]
    f = lib.oracle_attn_bwd_dropout
    f.restype = ci
    f.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, ci, ctypes.c_uint64, ctypes.c_uint64,
                  vp, ctypes.c_int64, vp, vp, vp, vp, ci]
    f = lib.oracle_attn_rows_ex
    f.restype = ci
    f.argtypes = [vp, vp, vp, ci, cf, cf, cf, ci, ci, ci, ci, ci, cf, ci, vp, ci, vp, ci, ci,
                  ctypes.c_uint64, ctypes.c_uint64, vp, ctypes.c_int64, vp, vp, ci]
    f = lib.oracle_attn_bwd_ex
    f.restype = ci
    f.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, vp, ci, vp, ci, ci, ctypes.c_uint64,
                  ctypes.c_uint64, vp, ctypes.c_int64, vp, vp, vp, vp, ci]
    f = lib.oracle_attn_bwd_keep
    f.restype = ci
    f.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, vp, ci, vp, ci, vp, ctypes.c_int64,
                  vp, vp, vp, vp, ci]
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library at ``path``."""
    path = path or LIBRARY
    with _lock:
        if path in _lib_cache:
            return _lib_cache[path]
        if path == LIBRARY:
            stale = (not os.path.exists(path)) or os.path.getmtime(path) < os.path.getmtime(SOURCE)
            if stale:
                compile_oracle()
        lib = _bind(ctypes.CDLL(path))
        _lib_cache[path] = lib
        return lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _as_bits(x: np.ndarray, name: str) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError(f"{name}: expected bf16 bit patterns as uint16, got {x.dtype}")
    return x


def _shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.shape != k.shape:
        raise ValueError("q must be [B,Hq,S,D]; k and v must both be [B,Hkv,S,D]")
    B, Hq, S, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    if (Bk, Sk, Dk) != (B, S, D):
        raise ValueError("q and k/v disagree on B, S or D")
    return B, Hq, Hkv, S, D


def _outputs(B, Hq, S, D, rows):
    if rows is None:
        return None, B * Hq * S, np.empty((B, Hq, S, D)), np.empty((B, Hq, S))
    rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    return rows_arr, rows_arr.size, np.empty((rows_arr.size, D)), np.empty((rows_arr.size,))


def attention_e4m3(q_codes, k_codes, v_codes, scale: float, descales=(1.0, 1.0, 1.0),
                   causal: bool = True, rows=None, nthreads: int | None = None,
                   lib: ctypes.CDLL | None = None):
    """As ``attention`` for FP8 E4M3 inputs: uint8 codes [B,H,S,D]; element value =
    decoded code * descale of its tensor (q, k, v)."""
    lib = lib or load()
    q, k, v = (np.ascontiguousarray(x) for x in (q_codes, k_codes, v_codes))
    for name, x in (("q", q), ("k", k), ("v", v)):
        if x.dtype != np.uint8:
            raise TypeError(f"{name}: expected E4M3 codes as uint8, got {x.dtype}")
    B, Hq, Hkv, S, D = _shapes(q, k, v)
    rows_arr, nrows, out, lse = _outputs(B, Hq, S, D, rows)
    dq, dk, dv = (ctypes.c_float(float(x)) for x in descales)
    rc = lib.oracle_attn_rows_e4m3(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, dq, dk, dv, B, Hq, Hkv, S, D,
        ctypes.c_float(scale), 1 if causal else 0,
        None if rows_arr is None else rows_arr.ctypes.data, nrows,
        out.ctypes.data, lse.ctypes.data, nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_attn_rows_e4m3 rejected its arguments")
    return out, lse


def attention_masked(q_bits, k_bits, v_bits, scale: float, block_mask, causal: bool = True,
                     rows=None, nthreads: int | None = None, lib: ctypes.CDLL | None = None):
    """As ``attention`` plus a block mask: uint8 [Hm, nt, nt] with nt = ceil(S/128)
    and Hm = 1 (shared by all heads) or Hq; entry 0 drops the 128 x 128 block of
    (query tile, key tile).  Rows without any visible key: O = 0, LSE = -inf."""
    lib = lib or load()
    q, k, v = (_as_bits(x, n) for x, n in ((q_bits, "q"), (k_bits, "k"), (v_bits, "v")))
    B, Hq, Hkv, S, D = _shapes(q, k, v)
    nt = (S + 127) // 128
    m = np.ascontiguousarray(block_mask, dtype=np.uint8)
    if m.ndim != 3 or m.shape[1:] != (nt, nt) or m.shape[0] not in (1, Hq):
        raise ValueError(f"block_mask must be [1 or Hq, {nt}, {nt}]")
    rows_arr, nrows, out, lse = _outputs(B, Hq, S, D, rows)
    rc = lib.oracle_attn_rows_masked(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, B, Hq, Hkv, S, D, ctypes.c_float(scale),
        1 if causal else 0, m.ctypes.data, m.shape[0],
        None if rows_arr is None else rows_arr.ctypes.data, nrows,
        out.ctypes.data, lse.ctypes.data, nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_attn_rows_masked rejected its arguments")
    return out, lse


def keep_row_bytes(S: int) -> int:
    """Bytes per query row of an element mask: 16 per 128 keys."""
    return 16 * ((S + 127) // 128)


def _keep(keep_bits, Hq: int, S: int) -> np.ndarray:
    m = np.ascontiguousarray(keep_bits, dtype=np.uint8)
    if m.ndim != 3 or m.shape[1:] != (S, keep_row_bytes(S)) or m.shape[0] not in (1, Hq):
        raise ValueError(f"keep_bits must be [1 or Hq, {S}, {keep_row_bytes(S)}]")
    return m


def _block(block_mask, Hq: int, S: int):
    if block_mask is None:
        return None
    nt = (S + 127) // 128
    m = np.ascontiguousarray(block_mask, dtype=np.uint8)
    if m.ndim != 3 or m.shape[1:] != (nt, nt) or m.shape[0] not in (1, Hq):
        raise ValueError(f"block_mask must be [1 or Hq, {nt}, {nt}]")
    return m


def attention_keep(q_bits, k_bits, v_bits, scale: float, keep_bits, causal: bool = True,
                   block_mask=None, rows=None, nthreads: int | None = None,
                   lib: ctypes.CDLL | None = None):
    """As ``attention`` plus an element mask: keep_bits uint8 [Hm, S, keep_row_bytes(S)],
    Hm = 1 or Hq; bit j % 8 of byte j / 8 of row i keeps key j for query i.  An
    optional block mask (as in ``attention_masked``) applies as well.  Rows
    without any visible key: O = 0, LSE = -inf."""
    lib = lib or load()
    q, k, v = (_as_bits(x, n) for x, n in ((q_bits, "q"), (k_bits, "k"), (v_bits, "v")))
    B, Hq, Hkv, S, D = _shapes(q, k, v)
    m = _keep(keep_bits, Hq, S)
    bm = _block(block_mask, Hq, S)
    rows_arr, nrows, out, lse = _outputs(B, Hq, S, D, rows)
    rc = lib.oracle_attn_rows_keep(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, B, Hq, Hkv, S, D, ctypes.c_float(scale),
        1 if causal else 0, m.ctypes.data, m.shape[0],
        None if bm is None else bm.ctypes.data, 1 if bm is None else bm.shape[0],
        None if rows_arr is None else rows_arr.ctypes.data, nrows,
        out.ctypes.data, lse.ctypes.data, nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_attn_rows_keep rejected its arguments")
    return out, lse


def attention_ex(q, k, v, scale: float, causal: bool = True, descales=None, block_mask=None,
                 keep_bits=None, dropout=None, rows=None, nthreads: int | None = None,
                 lib: ctypes.CDLL | None = None):
    """Every forward variant at once: q, k, v as bf16 bit patterns (uint16) or,
    with ``descales`` = (q, k, v) factors, E4M3 codes (uint8); optional block
    mask and keep bits (as in ``attention_masked`` / ``attention_keep``, both
    applying when given) and dropout = (p8, seed, offset)."""
    lib = lib or load()
    fp8 = descales is not None
    if fp8:
        q, k, v = (np.ascontiguousarray(x, dtype=np.uint8) for x in (q, k, v))
    else:
        q, k, v = (_as_bits(x, n) for x, n in ((q, "q"), (k, "k"), (v, "v")))
    B, Hq, Hkv, S, D = _shapes(q, k, v)
    bm = _block(block_mask, Hq, S)
    km = None if keep_bits is None else _keep(keep_bits, Hq, S)
    p8, seed, offset = dropout if dropout is not None else (0, 0, 0)
    ds = descales if fp8 else (1.0, 1.0, 1.0)
    rows_arr, nrows, out, lse = _outputs(B, Hq, S, D, rows)
    rc = lib.oracle_attn_rows_ex(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, 1 if fp8 else 0,
        *(ctypes.c_float(float(x)) for x in ds), B, Hq, Hkv, S, D, ctypes.c_float(scale),
        1 if causal else 0, None if bm is None else bm.ctypes.data, 1 if bm is None else bm.shape[0],
        None if km is None else km.ctypes.data, 1 if km is None else km.shape[0], int(p8),
        int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
        None if rows_arr is None else rows_arr.ctypes.data, nrows,
        out.ctypes.data, lse.ctypes.data, nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_attn_rows_ex rejected its arguments")
    return out, lse


def e4m3_decode(codes, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """The oracle's own E4M3 decoding of uint8 codes, as float64."""
    lib = lib or load()
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib.oracle_e4m3_decode(c.ctypes.data, c.size, out.ctypes.data)
    return out


def attention(q_bits, k_bits, v_bits, scale: float, causal: bool = True, rows=None,
              nthreads: int | None = None, lib: ctypes.CDLL | None = None):
    """O (float64) and LSE (float64, natural log) of causal scaled dot-product attention.

    q_bits: uint16 [B,Hq,S,D]; k_bits, v_bits: uint16 [B,Hkv,S,D] -- bf16 bit patterns.
    rows: optional int64 array of flat query-row ids (b*Hq + hq)*S + i; then the
          result has shape [len(rows), D] and [len(rows)].  Without rows the
          result is [B,Hq,S,D] and [B,Hq,S].
    """
    lib = lib or load()
    q_bits = _as_bits(q_bits, "q")
    k_bits = _as_bits(k_bits, "k")
    v_bits = _as_bits(v_bits, "v")
    if q_bits.ndim != 4 or k_bits.ndim != 4 or v_bits.shape != k_bits.shape:
        raise ValueError("q must be [B,Hq,S,D]; k and v must both be [B,Hkv,S,D]")
    B, Hq, S, D = q_bits.shape
    Bk, Hkv, Sk, Dk = k_bits.shape
    if (Bk, Sk, Dk) != (B, S, D):
        raise ValueError("q and k/v disagree on B, S or D")
    if rows is None:
        nrows = B * Hq * S
        rows_arr = None
        out_shape, lse_shape = (B, Hq, S, D), (B, Hq, S)
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.size
        out_shape, lse_shape = (nrows, D), (nrows,)
    out = np.empty(out_shape, dtype=np.float64)
    lse = np.empty(lse_shape, dtype=np.float64)
    nt = nthreads or default_threads()
    rc = lib.oracle_attn_rows(
        q_bits.ctypes.data, k_bits.ctypes.data, v_bits.ctypes.data,
        B, Hq, Hkv, S, D, ctypes.c_float(scale), 1 if causal else 0,
        None if rows_arr is None else rows_arr.ctypes.data, nrows,
        out.ctypes.data, lse.ctypes.data, nt,
    )
    if rc != 0:
        raise ValueError("oracle_attn_rows rejected its arguments")
    return out, lse


def attention_f64(q, k, v, scale: float, causal: bool = True, nthreads: int | None = None,
                  lib: ctypes.CDLL | None = None):
    """``attention`` on float64 inputs (no bf16 rounding), full [B,Hq,S,D] / [B,Hq,S] result."""
    lib = lib or load()
    q, k, v = (np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v))
    B, Hq, Hkv, S, D = _shapes(q, k, v)
    rows_arr, nrows, out, lse = _outputs(B, Hq, S, D, None)
    rc = lib.oracle_attn_rows_f64(q.ctypes.data, k.ctypes.data, v.ctypes.data, B, Hq, Hkv, S, D,
                                  ctypes.c_float(scale), 1 if causal else 0, None, nrows,
                                  out.ctypes.data, lse.ctypes.data, nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_attn_rows_f64 rejected its arguments")
    return out, lse


def attention_bwd(q, k, v, dout, scale: float, causal: bool = True, kv_heads=None,
                  nthreads: int | None = None, lib: ctypes.CDLL | None = None, block_mask=None,
                  keep_bits=None, dropout=None):
    """Gradients of the attention output: (dQ, dK, dV, delta) in float64.

    q, dout: [B,Hq,S,D]; k, v: [B,Hkv,S,D]; either all bf16 bit patterns
    (uint16) or all float64.  kv_heads: optional flat ids b*Hkv + hkv; then
    dQ and delta cover the G = Hq/Hkv query heads of each selected head,
    shapes [n, G, S, D] and [n, G, S], and dK, dV are [n, S, D].  Without
    kv_heads: dQ [B,Hq,S,D], dK and dV [B,Hkv,S,D], delta [B,Hq,S].
    delta_i = sum_j P_ij (dO_i . V_j), the row term of the softmax gradient.
    block_mask: optional uint8 [1 or Hq, nt, nt] as in ``attention_masked``;
    keep_bits: optional element mask as in ``attention_keep``.
    dropout: optional (p8, seed, offset) as in ``attention_dropout`` (masks may come with it).
    """
    lib = lib or load()
    f64 = np.asarray(q).dtype == np.float64
    conv = (lambda x, n: np.ascontiguousarray(x, dtype=np.float64)) if f64 else _as_bits
    q, k, v, dout = (conv(x, n) for x, n in ((q, "q"), (k, "k"), (v, "v"), (dout, "dout")))
    B, Hq, Hkv, S, D = _shapes(q, k, v)
    if dout.shape != q.shape:
        raise ValueError("dout must have the shape of q")
    G = Hq // Hkv
    if kv_heads is None:
        heads, n = None, B * Hkv
        dq_shape, kv_shape, d_shape = (B, Hq, S, D), (B, Hkv, S, D), (B, Hq, S)
    else:
        heads = np.ascontiguousarray(np.asarray(kv_heads, dtype=np.int64))
        n = heads.size
        dq_shape, kv_shape, d_shape = (n, G, S, D), (n, S, D), (n, G, S)
    dq, dk, dv = np.empty(dq_shape), np.empty(kv_shape), np.empty(kv_shape)
    delta = np.empty(d_shape)
    common = (q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, 1 if f64 else 0, B, Hq,
              Hkv, S, D, ctypes.c_float(scale), 1 if causal else 0)
    tail = (None if heads is None else heads.ctypes.data, n, dq.ctypes.data, dk.ctypes.data,
            dv.ctypes.data, delta.ctypes.data, nthreads or default_threads())
    bm = _block(block_mask, Hq, S)
    if dropout is not None and (bm is not None or keep_bits is not None):
        km = None if keep_bits is None else _keep(keep_bits, Hq, S)
        p8, seed, offset = dropout
        rc = lib.oracle_attn_bwd_ex(*common, None if bm is None else bm.ctypes.data,
                                    1 if bm is None else bm.shape[0],
                                    None if km is None else km.ctypes.data,
                                    1 if km is None else km.shape[0], int(p8),
                                    int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), *tail)
    elif dropout is not None:
        p8, seed, offset = dropout
        rc = lib.oracle_attn_bwd_dropout(*common, int(p8), int(seed) & (2**64 - 1),
                                         int(offset) & (2**64 - 1), *tail)
    elif keep_bits is not None:
        km = _keep(keep_bits, Hq, S)
        rc = lib.oracle_attn_bwd_keep(*common, km.ctypes.data, km.shape[0],
                                      None if bm is None else bm.ctypes.data,
                                      1 if bm is None else bm.shape[0], *tail)
    elif bm is None:
        rc = lib.oracle_attn_bwd(*common, *tail)
    else:
        rc = lib.oracle_attn_bwd_masked(*common, bm.ctypes.data, bm.shape[0], *tail)
    if rc != 0:
        raise ValueError("oracle_attn_bwd rejected its arguments")
    return dq, dk, dv, delta


def attention_dropout(q_bits, k_bits, v_bits, scale: float, p8: int, seed: int, offset: int,
                      causal: bool = True, rows=None, nthreads: int | None = None,
                      lib: ctypes.CDLL | None = None):
    """``attention`` with dropout of the weights: each dropped with probability
    p8/256 by Philox4x32-10 (key from the 64-bit seed, the 32-bit offset in the
    counter), kept ones scaled by 256/(256-p8).  The LSE is that of the
    undropped softmax."""
    lib = lib or load()
    q, k, v = (_as_bits(x, n) for x, n in ((q_bits, "q"), (k_bits, "k"), (v_bits, "v")))
    B, Hq, Hkv, S, D = _shapes(q, k, v)
    rows_arr, nrows, out, lse = _outputs(B, Hq, S, D, rows)
    rc = lib.oracle_attn_rows_dropout(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, B, Hq, Hkv, S, D, ctypes.c_float(scale),
        1 if causal else 0, int(p8), ctypes.c_uint64(seed), ctypes.c_uint64(offset),
        None if rows_arr is None else rows_arr.ctypes.data, nrows, out.ctypes.data,
        lse.ctypes.data, nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_attn_rows_dropout rejected its arguments")
    return out, lse


def philox4x32(ctr, key, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """The oracle's Philox4x32-10 block for one counter (4 x uint32) and key (2 x uint32)."""
    lib = lib or load()
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.empty(4, dtype=np.uint32)
    lib.oracle_philox4x32(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return out


def out_proj(o, w, bias=None) -> np.ndarray:
    """The attention output projection, in float64: Y[b, s, e] = sum over
    k = h*D + d of O[b, h, s, d] * W[e, k] (+ bias[e]).

    o: [B, H, S, D] and w: [E, H*D] as bf16 bit patterns (uint16) or floats;
    bias: [E] or None.  Written as its definition -- the heads of each position
    laid side by side into one H*D row (the concatenation that precedes the
    projection), times W^T -- with numpy's float64 matmul as the one library step.
    """
    def wide(x):
        x = np.asarray(x)
        if x.dtype == np.uint16:
            return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
        return x.astype(np.float64)
    O, W = wide(o), wide(w)
    B, H, S, D = O.shape
    if W.ndim != 2 or W.shape[1] != H * D:
        raise ValueError("w must be [E, H*D]")
    rows = O.transpose(0, 2, 1, 3).reshape(B, S, H * D)  # [b, s, h*D + d]
    Y = rows @ W.T
    if bias is not None:
        Y = Y + np.asarray(bias, dtype=np.float64)
    return Y
