"""Seeded synthetic inputs: i.i.d. Gaussian values rounded to bf16.

This module holds none of the attention arithmetic.  It is the one piece of
code that both the CUDA path's callers and the CPU oracle's callers share, so
that both sides see the same bits.

The pages profile attention on ``torch.randn`` inputs of shape
[B, H, S, D] (the ai-manual.ru article, section 1); the values here are the
same distribution, N(0, 1) times a per-workload ``sigma``, drawn from a
counter-based generator so the bits do not depend on the host (x86_64 or
aarch64) or on library versions:

* uniform bits: SplitMix64 (Steele, Lea and Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014) applied to a per-tensor key
  plus the element counter;
* normals: the Box-Muller transform (Box and Muller, 1958) in float64;
* rounding: float64 -> float32 (numpy, round to nearest even), then
  float32 -> bf16 by round-to-nearest-even on the bit pattern.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22  # elements per work item


def _splitmix64(x: np.ndarray) -> np.ndarray:
    """SplitMix64 output function of state ``x`` (uint64, wrapping arithmetic)."""
    z = x.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def _tensor_key(seed: int, stream: int) -> np.uint64:
    base = np.array([(seed * 0x100000001B3 + stream * 0x1F123BB5) & 0xFFFFFFFFFFFFFFFF],
                    dtype=np.uint64)
    return _splitmix64(base)[0]


def _normals_chunk(key: np.uint64, start: int, count: int) -> np.ndarray:
    """Normals with element index start .. start+count-1 of the stream ``key``."""
    npairs = (count + 1) // 2
    first_pair = start // 2
    pair_idx = np.arange(first_pair, first_pair + npairs + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        c0 = key + (np.uint64(2) * pair_idx + np.uint64(1)) * _GOLDEN
        c1 = key + (np.uint64(2) * pair_idx + np.uint64(2)) * _GOLDEN
        u0 = _splitmix64(c0)
        u1 = _splitmix64(c1)
    # 53-bit uniforms: a in (0, 1], b in [0, 1)
    a = ((u0 >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)
    b = (u1 >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    r = np.sqrt(-2.0 * np.log(a))
    t = 2.0 * np.pi * b
    pairs = np.empty((pair_idx.size, 2), dtype=np.float64)
    pairs[:, 0] = r * np.cos(t)
    pairs[:, 1] = r * np.sin(t)
    flat = pairs.reshape(-1)
    off = start - 2 * first_pair
    return flat[off:off + count]


def float32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits.

    NaN is not expected here (Gaussian draws are finite) and is not special-cased.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = u + np.uint64(0x7FFF) + lsb
    return (u >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_float32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def gaussian_bf16(shape, seed: int, stream: int, sigma: float = 1.0,
                  threads: int | None = None) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0, sigma^2) draws, deterministic in (seed, stream)."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    out = np.empty(n, dtype=np.uint16)
    key = _tensor_key(seed, stream)

    def work(start: int) -> None:
        cnt = min(_CHUNK, n - start)
        x = _normals_chunk(key, start, cnt)
        if sigma != 1.0:
            x = x * sigma
        out[start:start + cnt] = float32_to_bf16_bits(x.astype(np.float32))

    starts = list(range(0, n, _CHUNK))
    nthreads = threads or min(len(starts), max(1, min(16, os.cpu_count() or 1)))
    if nthreads <= 1 or len(starts) <= 1:
        for s in starts:
            work(s)
    else:
        with ThreadPoolExecutor(max_workers=nthreads) as ex:
            list(ex.map(work, starts))
    return out.reshape(shape)


def qkv_bf16(B: int, Hq: int, Hkv: int, S: int, D: int, seed: int, sigma: float = 1.0):
    """Q [B,Hq,S,D], K and V [B,Hkv,S,D] as bf16 bit patterns, drawn in the order q, k, v."""
    q = gaussian_bf16((B, Hq, S, D), seed, 0, sigma)
    k = gaussian_bf16((B, Hkv, S, D), seed, 1, sigma)
    v = gaussian_bf16((B, Hkv, S, D), seed, 2, sigma)
    return q, k, v


def float32_to_e4m3_codes(x: np.ndarray) -> np.ndarray:
    """Round float32 values to FP8 E4M3 (nearest, ties to even, saturating at
    +-448 like PyTorch's float8_e4m3fn conversion); returns uint8 codes."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    t = t.clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


def gaussian_e4m3(shape, seed: int, stream: int, sigma: float = 1.0) -> np.ndarray:
    """E4M3 codes (uint8) of N(0, sigma^2) draws: the bf16 draws of the same
    (seed, stream), widened, then rounded to E4M3."""
    return float32_to_e4m3_codes(bf16_bits_to_float32(gaussian_bf16(shape, seed, stream, sigma)))


def qkv_e4m3(B: int, Hq: int, Hkv: int, S: int, D: int, seed: int, sigma: float = 1.0):
    """Q [B,Hq,S,D], K and V [B,Hkv,S,D] as E4M3 codes, drawn in the order q, k, v."""
    q = gaussian_e4m3((B, Hq, S, D), seed, 0, sigma)
    k = gaussian_e4m3((B, Hkv, S, D), seed, 1, sigma)
    v = gaussian_e4m3((B, Hkv, S, D), seed, 2, sigma)
    return q, k, v


def random_block_mask(mask_heads: int, S: int, density: float, seed: int,
                      stream: int = 7) -> np.ndarray:
    """uint8 [mask_heads, nt, nt] (nt = ceil(S/128)) with each entry 1 with
    probability ``density``, from the same SplitMix64 stream construction as
    the value draws: entry e keeps its block when its 53-bit uniform < density."""
    nt = (int(S) + 127) // 128
    n = int(mask_heads) * nt * nt
    key = _tensor_key(seed, stream)
    with np.errstate(over="ignore"):
        u = _splitmix64(key + (np.arange(n, dtype=np.uint64) + np.uint64(1)) * _GOLDEN)
    uniform = (u >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    return (uniform < density).astype(np.uint8).reshape(mask_heads, nt, nt)


def keep_row_bytes(S: int) -> int:
    """Bytes per query row of an element mask: 16 per 128 keys."""
    return 16 * ((int(S) + 127) // 128)


def pack_keep_bits(keep: np.ndarray) -> np.ndarray:
    """bool [Hm, S, S] (query, key) -> uint8 [Hm, S, keep_row_bytes(S)]: bit
    j % 8 of byte j / 8 of row i set when key j is kept for query i; the
    padding bits past key S-1 are 0."""
    keep = np.asarray(keep, dtype=bool)
    Hm, S, S2 = keep.shape
    if S2 != S:
        raise ValueError("keep must be [Hm, S, S]")
    padded = np.zeros((Hm, S, keep_row_bytes(S) * 8), dtype=bool)
    padded[:, :, :S] = keep
    return np.packbits(padded, axis=-1, bitorder="little")


def unpack_keep_bits(bits: np.ndarray, S: int) -> np.ndarray:
    """Inverse of ``pack_keep_bits``: bool [Hm, S, S]."""
    return np.unpackbits(np.asarray(bits, dtype=np.uint8), axis=-1, bitorder="little")[:, :, :S].astype(bool)


def random_keep_bits(mask_heads: int, S: int, density: float, seed: int,
                     stream: int = 9) -> np.ndarray:
    """Element mask with each (query, key) pair kept with probability
    ``density`` (53-bit SplitMix64 uniforms as in ``random_block_mask``),
    packed as ``pack_keep_bits`` does."""
    n = int(mask_heads) * int(S) * int(S)
    key = _tensor_key(seed, stream)
    with np.errstate(over="ignore"):
        u = _splitmix64(key + (np.arange(n, dtype=np.uint64) + np.uint64(1)) * _GOLDEN)
    uniform = (u >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    return pack_keep_bits((uniform < density).reshape(mask_heads, S, S))


def window_keep_bits(S: int, window: int) -> np.ndarray:
    """Local (sliding-window) element mask shared by all heads: query i keeps
    keys i - window < j <= i, packed as ``pack_keep_bits`` does."""
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    return pack_keep_bits(((j <= i) & (j > i - window))[None])


def block_mask_of_keep_bits(bits: np.ndarray, S: int) -> np.ndarray:
    """uint8 [Hm, nt, nt]: 1 where the 128 x 128 (query tile, key tile) block
    of the element mask keeps at least one pair, so that a kernel may skip the
    other blocks without changing the result."""
    bits = np.asarray(bits, dtype=np.uint8)
    Hm = bits.shape[0]
    nt = (int(S) + 127) // 128
    rows = np.zeros((Hm, nt * 128, bits.shape[2]), dtype=np.uint8)
    rows[:, :S] = bits
    per_tile = rows.reshape(Hm, nt, 128, nt, 16).any(axis=(2, 4))
    return per_tile.astype(np.uint8)
