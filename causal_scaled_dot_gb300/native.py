"""ctypes binding of libattn (include/attn.h): argument marshalling only.

Every step of the attention forward runs in the CUDA library; this module
turns PyTorch tensors (or raw integers) into the pointers, sizes and stream
handle the C ABI takes, and turns return codes into exceptions.  There is no
CPU path: if the library cannot be built or loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import threading

from . import build as _build

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_MISALIGNED = 3
ATTN_ERR_DEVICE = 4
ATTN_ERR_LAUNCH = 5
ATTN_ERR_TIMEOUT = 6

_lock = threading.Lock()
_lib: ctypes.CDLL | None = None


class AttnError(RuntimeError):
    """A non-zero return code from libattn."""

    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {attn_status_string(code)} (code {code})")


def load() -> ctypes.CDLL:
    """Build libattn.so if it is missing or older than its sources, then load it."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build()  # raises if nvcc fails: no fallback
        lib = ctypes.CDLL(path)
        vp, ci = ctypes.c_void_p, ctypes.c_int
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ctypes.c_float, ci, vp]
        lib.attn_fwd.restype = ci
        cf = ctypes.c_float
        lib.attn_fwd_block_masked.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, vp, ci,
                                              vp]
        lib.attn_fwd_block_masked.restype = ci
        lib.attn_fwd_elem_masked.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, vp, ci,
                                             vp, ci, vp]
        lib.attn_fwd_elem_masked.restype = ci
        lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci,
                                 vp]
        lib.attn_bwd.restype = ci
        lib.attn_bwd_block_masked.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci,
                                              ci, cf, ci, vp, ci, vp]
        lib.attn_bwd_block_masked.restype = ci
        lib.attn_bwd_elem_masked.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci,
                                             ci, cf, ci, vp, ci, vp, ci, vp]
        lib.attn_bwd_elem_masked.restype = ci
        lib.attn_bwd_dropout.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf,
                                         ci, cf, ctypes.c_ulonglong, ctypes.c_ulonglong, vp]
        lib.attn_bwd_dropout.restype = ci
        opts_p = ctypes.POINTER(AttnOptions)
        lib.attn_fwd_ex.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, opts_p, vp]
        lib.attn_fwd_ex.restype = ci
        lib.attn_bwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci,
                                    opts_p, vp]
        lib.attn_bwd_ex.restype = ci
        u64 = ctypes.c_ulonglong
        lib.attn_fwd_dropout.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, cf, u64, u64,
                                         vp]
        lib.attn_fwd_dropout.restype = ci
        lib.attn_out_proj.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, vp]
        lib.attn_out_proj.restype = ci
        lib.attn_fwd_fp8.argtypes = [vp, vp, vp, cf, cf, cf, vp, vp, ci, ci, ci, ci, ci, cf, ci, vp]
        lib.attn_fwd_fp8.restype = ci
        lib.attn_sync_status.argtypes = [vp]
        lib.attn_sync_status.restype = ci
        lib.attn_selftest_wait_timeout.argtypes = [ci, vp]
        lib.attn_selftest_wait_timeout.restype = ci
        lib.attn_status_string.argtypes = [ci]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_version.argtypes = []
        lib.attn_version.restype = ci
        u16p = ctypes.POINTER(ctypes.c_ushort)
        lib.attn_fwd_schedule.argtypes = [ci, ci, ci, ci, u16p, u16p]
        lib.attn_fwd_schedule.restype = ci
        _lib = lib
        return lib


def library_path() -> str:
    return _build.LIBRARY


class AttnOptions(ctypes.Structure):
    """The C struct attn_options_t (include/attn.h), field for field."""
    _fields_ = [("input_format", ctypes.c_int), ("q_descale", ctypes.c_float),
                ("k_descale", ctypes.c_float), ("v_descale", ctypes.c_float),
                ("block_mask", ctypes.c_void_p), ("mask_heads", ctypes.c_int),
                ("keep_bits", ctypes.c_void_p), ("keep_heads", ctypes.c_int),
                ("dropout_p", ctypes.c_float), ("seed", ctypes.c_ulonglong),
                ("offset", ctypes.c_ulonglong)]


ATTN_INPUT_BF16, ATTN_INPUT_E4M3 = 0, 1


def options(e4m3_descales=None, block_mask=None, keep_bits=None, dropout_p: float = 0.0, seed: int = 0,
            offset: int = 0) -> AttnOptions:
    """An attn_options_t: E4M3 inputs when ``e4m3_descales`` = (q, k, v) is given; masks
    as CUDA uint8 tensors (their first dimension gives mask_heads / keep_heads).  The
    returned object also holds the mask tensors, which keeps them alive while it is in
    use and lets the entry points check their sizes (a mask given as an int pointer must
    be kept alive by the caller)."""
    o = AttnOptions()
    o.tensors = (block_mask, keep_bits)
    o.input_format = ATTN_INPUT_E4M3 if e4m3_descales is not None else ATTN_INPUT_BF16
    o.q_descale, o.k_descale, o.v_descale = e4m3_descales if e4m3_descales is not None else (1.0, 1.0, 1.0)
    o.block_mask = _ptr(block_mask)
    o.mask_heads = 1 if block_mask is None else int(block_mask.shape[0])
    o.keep_bits = _ptr(keep_bits)
    o.keep_heads = 1 if keep_bits is None else int(keep_bits.shape[0])
    o.dropout_p = float(dropout_p)
    o.seed = int(seed) & (2**64 - 1)
    o.offset = int(offset) & (2**64 - 1)
    return o


def _sizes(*items):
    """Raise ValueError when a tensor argument holds fewer bytes than the sizes
    passed with it imply: the C entry points read and write exactly that many
    bytes from the addresses they receive and cannot check them.  ``items`` are
    (name, tensor / int pointer / None, bytes needed); only tensors are checked."""
    for name, x, need in items:
        if hasattr(x, "element_size") and hasattr(x, "numel"):
            have = int(x.numel()) * int(x.element_size())
            if need > 0 and have < need:
                raise ValueError(f"{name} holds {have} bytes; the sizes given need {need}")


def _attn_bytes(B, Hq, Hkv, S, D, in_bytes=2):
    """Bytes of q, of k (= v), of out (= dout, dq) and of lse (= delta)."""
    return (B * Hq * S * D * in_bytes, B * Hkv * S * D * in_bytes, B * Hq * S * D * 2, B * Hq * S * 4)


def _mask_bytes(S, mask_heads=1, keep_heads=1):
    """Bytes of a block mask [mask_heads, nt, nt] and of keep bits [keep_heads, S, 16 nt]."""
    nt = -(-S // 128)
    return mask_heads * nt * nt, keep_heads * S * 16 * nt


def _fwd_sizes(q, k, v, out, lse, B, Hq, Hkv, S, D, in_bytes=2, block_mask=None, mask_heads=1,
               keep_bits=None, keep_heads=1):
    qb, kb, ob, lb = _attn_bytes(B, Hq, Hkv, S, D, in_bytes)
    mb, eb = _mask_bytes(S, mask_heads, keep_heads)
    _sizes(("q", q, qb), ("k", k, kb), ("v", v, kb), ("out", out, ob), ("lse", lse, lb),
           ("block_mask", block_mask, mb), ("keep_bits", keep_bits, eb))


def _bwd_sizes(q, k, v, out, dout, lse, delta, dq, dk, dv, B, Hq, Hkv, S, D, block_mask=None,
               mask_heads=1, keep_bits=None, keep_heads=1):
    qb, kb, ob, lb = _attn_bytes(B, Hq, Hkv, S, D)
    mb, eb = _mask_bytes(S, mask_heads, keep_heads)
    _sizes(("q", q, qb), ("k", k, kb), ("v", v, kb), ("out", out, ob), ("dout", dout, ob), ("lse", lse, lb),
           ("delta", delta, lb), ("dq", dq, ob), ("dk", dk, kb), ("dv", dv, kb),
           ("block_mask", block_mask, mb), ("keep_bits", keep_bits, eb))


def _opts_masks(opts):
    """The mask tensors an AttnOptions holds and still points at (None otherwise)."""
    if opts is None:
        return None, None
    held = getattr(opts, "tensors", (None, None))
    addr = (opts.block_mask, opts.keep_bits)
    return tuple(t if t is not None and hasattr(t, "data_ptr") and a and t.data_ptr() == a else None
                 for t, a in zip(held, addr))


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    import torch
    if isinstance(x, torch.Tensor):
        if not x.is_cuda:
            raise ValueError("tensor arguments must live in CUDA device memory")
        if not x.is_contiguous():
            raise ValueError("tensor arguments must be contiguous (the C ABI takes dense layouts)")
        return x.data_ptr()
    raise TypeError(f"expected a CUDA tensor, an int pointer or None, got {type(x)!r}")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    handle = getattr(s, "cuda_stream", None)
    if handle is None:
        raise TypeError(f"expected a torch.cuda.Stream, an int handle or None, got {type(s)!r}")
    return handle


def attn_fwd(q, k, v, out, lse, B: int, Hq: int, Hkv: int, S: int, D: int, scale: float,
             causal: bool | int, stream=None, check: bool = True) -> int:
    """The C entry point ``attn_fwd`` with the same argument order.

    Tensors may be CUDA tensors (their data pointers are passed) or raw device
    pointers as ints; ``lse`` may be None.  ``stream`` defaults to PyTorch's
    current stream.  Raises AttnError on a non-zero code unless check=False.
    """
    _fwd_sizes(q, k, v, out, lse, int(B), int(Hq), int(Hkv), int(S), int(D))
    rc = load().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), int(B), int(Hq),
                         int(Hkv), int(S), int(D), float(scale), 1 if causal else 0,
                         _stream(stream))
    if check and rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd")
    return rc


def attn_fwd_block_masked(q, k, v, out, lse, B: int, Hq: int, Hkv: int, S: int, D: int,
                          scale: float, causal: bool | int, block_mask, mask_heads: int, stream=None,
                          check: bool = True) -> int:
    """The C entry point ``attn_fwd_block_masked``: ``block_mask`` is a uint8 CUDA
    tensor (or device pointer) [mask_heads, ceil(S/128), ceil(S/128)]."""
    _fwd_sizes(q, k, v, out, lse, int(B), int(Hq), int(Hkv), int(S), int(D), block_mask=block_mask,
               mask_heads=int(mask_heads))
    rc = load().attn_fwd_block_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), int(B),
                                      int(Hq), int(Hkv), int(S), int(D), float(scale),
                                      1 if causal else 0, _ptr(block_mask), int(mask_heads),
                                      _stream(stream))
    if check and rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_block_masked")
    return rc


def attn_fwd_elem_masked(q, k, v, out, lse, B: int, Hq: int, Hkv: int, S: int, D: int,
                         scale: float, causal: bool | int, keep_bits, keep_heads: int,
                         block_mask=None, mask_heads: int = 1, stream=None,
                         check: bool = True) -> int:
    """The C entry point ``attn_fwd_elem_masked``: ``keep_bits`` is a uint8 CUDA
    tensor (or device pointer) [keep_heads, S, 16*ceil(S/128)] of keep bits;
    ``block_mask`` optional as in ``attn_fwd_block_masked``."""
    _fwd_sizes(q, k, v, out, lse, int(B), int(Hq), int(Hkv), int(S), int(D), block_mask=block_mask,
               mask_heads=int(mask_heads), keep_bits=keep_bits, keep_heads=int(keep_heads))
    rc = load().attn_fwd_elem_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), int(B),
                                     int(Hq), int(Hkv), int(S), int(D), float(scale),
                                     1 if causal else 0, _ptr(keep_bits), int(keep_heads),
                                     _ptr(block_mask), int(mask_heads), _stream(stream))
    if check and rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_elem_masked")
    return rc


def attn_fwd_dropout(q, k, v, out, lse, B: int, Hq: int, Hkv: int, S: int, D: int, scale: float,
                     causal: bool | int, dropout_p: float, seed: int, offset: int, stream=None,
                     check: bool = True) -> int:
    """The C entry point ``attn_fwd_dropout`` (drop probability rounded to p8/256)."""
    _fwd_sizes(q, k, v, out, lse, int(B), int(Hq), int(Hkv), int(S), int(D))
    rc = load().attn_fwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), int(B), int(Hq),
                                 int(Hkv), int(S), int(D), float(scale), 1 if causal else 0,
                                 float(dropout_p), int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                                 _stream(stream))
    if check and rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_dropout")
    return rc


def attn_out_proj(out, w, bias, y, B: int, H: int, S: int, D: int, E: int, stream=None,
                  check: bool = True) -> int:
    """The C entry point ``attn_out_proj``: Y = concat_heads(O) W^T + bias."""
    B, H, S, D, E = int(B), int(H), int(S), int(D), int(E)
    _sizes(("out", out, B * H * S * D * 2), ("w", w, E * H * D * 2), ("bias", bias, E * 4),
           ("y", y, B * S * E * 2))
    rc = load().attn_out_proj(_ptr(out), _ptr(w), _ptr(bias), _ptr(y), int(B), int(H), int(S), int(D),
                              int(E), _stream(stream))
    if check and rc != ATTN_OK:
        raise AttnError(rc, "attn_out_proj")
    return rc


def attn_bwd(q, k, v, out, dout, lse, delta, dq, dk, dv, B: int, Hq: int, Hkv: int, S: int, D: int,
             scale: float, causal: bool | int, stream=None, check: bool = True) -> int:
    """The C entry point ``attn_bwd``: dQ, dK, dV (and delta) for upstream dO."""
    _bwd_sizes(q, k, v, out, dout, lse, delta, dq, dk, dv, int(B), int(Hq), int(Hkv), int(S), int(D))
    rc = load().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(delta),
                         _ptr(dq), _ptr(dk), _ptr(dv), int(B), int(Hq), int(Hkv), int(S), int(D),
                         float(scale), 1 if causal else 0, _stream(stream))
    if check and rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd")
    return rc


def attn_bwd_block_masked(q, k, v, out, dout, lse, delta, dq, dk, dv, B: int, Hq: int, Hkv: int,
                          S: int, D: int, scale: float, causal: bool | int, block_mask, mask_heads: int,
                          stream=None, check: bool = True) -> int:
    """The C entry point ``attn_bwd_block_masked`` (the mask of the forward call)."""
    _bwd_sizes(q, k, v, out, dout, lse, delta, dq, dk, dv, int(B), int(Hq), int(Hkv), int(S), int(D),
               block_mask=block_mask, mask_heads=int(mask_heads))
    rc = load().attn_bwd_block_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                                      _ptr(delta), _ptr(dq), _ptr(dk), _ptr(dv), int(B), int(Hq),
                                      int(Hkv), int(S), int(D), float(scale), 1 if causal else 0,
                                      _ptr(block_mask), int(mask_heads), _stream(stream))
    if check and rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd_block_masked")
    return rc


def attn_bwd_elem_masked(q, k, v, out, dout, lse, delta, dq, dk, dv, B: int, Hq: int, Hkv: int,
                         S: int, D: int, scale: float, causal: bool | int, keep_bits,
                         keep_heads: int, block_mask=None, mask_heads: int = 1, stream=None,
                         check: bool = True) -> int:
    """The C entry point ``attn_bwd_elem_masked`` (masks as in ``attn_fwd_elem_masked``)."""
    _bwd_sizes(q, k, v, out, dout, lse, delta, dq, dk, dv, int(B), int(Hq), int(Hkv), int(S), int(D),
               block_mask=block_mask, mask_heads=int(mask_heads), keep_bits=keep_bits,
               keep_heads=int(keep_heads))
    rc = load().attn_bwd_elem_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                                     _ptr(delta), _ptr(dq), _ptr(dk), _ptr(dv), int(B), int(Hq),
                                     int(Hkv), int(S), int(D), float(scale), 1 if causal else 0,
                                     _ptr(keep_bits), int(keep_heads), _ptr(block_mask),
                                     int(mask_heads), _stream(stream))
    if check and rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd_elem_masked")
    return rc


def attn_bwd_dropout(q, k, v, out, dout, lse, delta, dq, dk, dv, B: int, Hq: int, Hkv: int, S: int,
                     D: int, scale: float, causal: bool | int, dropout_p: float, seed: int, offset: int,
                     stream=None, check: bool = True) -> int:
    """The C entry point ``attn_bwd_dropout`` (the dropout of the forward call)."""
    _bwd_sizes(q, k, v, out, dout, lse, delta, dq, dk, dv, int(B), int(Hq), int(Hkv), int(S), int(D))
    rc = load().attn_bwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                                 _ptr(delta), _ptr(dq), _ptr(dk), _ptr(dv), int(B), int(Hq), int(Hkv),
                                 int(S), int(D), float(scale), 1 if causal else 0, float(dropout_p),
                                 int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), _stream(stream))
    if check and rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd_dropout")
    return rc


def attn_fwd_ex(q, k, v, out, lse, B: int, Hq: int, Hkv: int, S: int, D: int, scale: float,
                causal: bool | int, opts: AttnOptions | None, stream=None, check: bool = True) -> int:
    """The C entry point ``attn_fwd_ex`` (``opts`` from ``options``, or None)."""
    bm, kb = _opts_masks(opts)
    _fwd_sizes(q, k, v, out, lse, int(B), int(Hq), int(Hkv), int(S), int(D),
               in_bytes=1 if opts is not None and opts.input_format == ATTN_INPUT_E4M3 else 2,
               block_mask=bm, mask_heads=opts.mask_heads if bm is not None else 1,
               keep_bits=kb, keep_heads=opts.keep_heads if kb is not None else 1)
    rc = load().attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), int(B), int(Hq), int(Hkv),
                            int(S), int(D), float(scale), 1 if causal else 0,
                            None if opts is None else ctypes.byref(opts), _stream(stream))
    if check and rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_ex")
    return rc


def attn_bwd_ex(q, k, v, out, dout, lse, delta, dq, dk, dv, B: int, Hq: int, Hkv: int, S: int, D: int,
                scale: float, causal: bool | int, opts: AttnOptions | None, stream=None,
                check: bool = True) -> int:
    """The C entry point ``attn_bwd_ex`` (``opts`` as given to ``attn_fwd_ex``)."""
    bm, kb = _opts_masks(opts)
    _bwd_sizes(q, k, v, out, dout, lse, delta, dq, dk, dv, int(B), int(Hq), int(Hkv), int(S), int(D),
               block_mask=bm, mask_heads=opts.mask_heads if bm is not None else 1,
               keep_bits=kb, keep_heads=opts.keep_heads if kb is not None else 1)
    rc = load().attn_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(delta),
                            _ptr(dq), _ptr(dk), _ptr(dv), int(B), int(Hq), int(Hkv), int(S), int(D),
                            float(scale), 1 if causal else 0, None if opts is None else ctypes.byref(opts),
                            _stream(stream))
    if check and rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd_ex")
    return rc


def attn_fwd_fp8(q, k, v, q_descale: float, k_descale: float, v_descale: float, out, lse, B: int,
                 Hq: int, Hkv: int, S: int, D: int, scale: float, causal: bool | int, stream=None,
                 check: bool = True) -> int:
    """The C entry point ``attn_fwd_fp8`` (E4M3 inputs with per-tensor descales),
    same argument order; tensors or raw device pointers as in ``attn_fwd``."""
    _fwd_sizes(q, k, v, out, lse, int(B), int(Hq), int(Hkv), int(S), int(D), in_bytes=1)
    rc = load().attn_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), float(q_descale), float(k_descale),
                             float(v_descale), _ptr(out), _ptr(lse), int(B), int(Hq), int(Hkv),
                             int(S), int(D), float(scale), 1 if causal else 0, _stream(stream))
    if check and rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_fp8")
    return rc


def attn_sync_status(stream=None, check: bool = True) -> int:
    rc = load().attn_sync_status(_stream(stream))
    if check and rc != ATTN_OK:
        raise AttnError(rc, "attn_sync_status")
    return rc


def attn_selftest_wait_timeout(limit_us: int, stream=None) -> int:
    return load().attn_selftest_wait_timeout(int(limit_us), _stream(stream))


def attn_status_string(code: int) -> str:
    try:
        return load().attn_status_string(int(code)).decode()
    except Exception:  # pragma: no cover - message of last resort
        return f"status {code}"


def attn_version() -> int:
    return load().attn_version()


def fwd_schedule(batch_heads: int, num_q_tiles: int, causal: bool, num_ctas: int):
    """The forward kernel's work order (``attn_fwd_schedule``): a list with, for
    each CTA, the unit numbers it runs in turn; None when the kernel falls back
    to its arithmetic order for this shape."""
    import numpy as np
    npairs = (num_q_tiles + 1) // 2
    order = np.zeros(max(batch_heads * npairs, 1), dtype=np.uint16)
    start = np.zeros(num_ctas + 1, dtype=np.uint16)
    u16p = ctypes.POINTER(ctypes.c_ushort)
    rc = load().attn_fwd_schedule(int(batch_heads), int(num_q_tiles), 1 if causal else 0, int(num_ctas),
                                  order.ctypes.data_as(u16p), start.ctypes.data_as(u16p))
    if rc == ATTN_ERR_UNSUPPORTED:
        return None
    if rc != ATTN_OK:
        raise ValueError(attn_status_string(rc))
    return [order[start[c]:start[c + 1]].astype(int).tolist() for c in range(num_ctas)]


def _check_attention_tensors(named):
    """Validate the tensors of ``attention`` / ``attention_trainable`` before any
    library call: bf16 q, k, v that are contiguous 4-D CUDA tensors, and every
    tensor given (outputs and masks included) on one and the same device.  The C
    ABI runs on the calling thread's current device, so a tensor on another GPU
    would hand that device's addresses to a kernel launched elsewhere.  Returns
    that device."""
    import torch
    device = None
    for name, t in named:
        if t is None:
            continue
        if name in ("q", "k", "v"):
            if not getattr(t, "is_cuda", False) or t.dtype != torch.bfloat16:
                raise ValueError(f"{name} must be a bf16 CUDA tensor")
            if t.dim() != 4 or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous [B,H,S,D] tensor")
        elif not getattr(t, "is_cuda", False):
            raise ValueError(f"{name} must be a CUDA tensor")
        if device is None:
            device = t.device
        elif t.device != device:
            raise ValueError(f"{name} is on {t.device} but q is on {device}: all tensors of one call "
                             "must be on the same device")
    return device


def _device_stream(device, stream):
    """The stream to launch on: the one given, else the current stream of ``device``."""
    import torch
    return torch.cuda.current_stream(device) if stream is None else stream


def attention(q, k, v, causal: bool = True, scale: float | None = None, out=None, lse=None,
              return_lse: bool = True, stream=None, check_status: bool = False):
    """O (and LSE) for CUDA tensors q [B,Hq,S,D], k/v [B,Hkv,S,D] in bf16.

    Allocates ``out`` (bf16 [B,Hq,S,D]) and ``lse`` (fp32 [B,Hq,S]) with
    PyTorch when they are not given, checks dtypes, shapes, contiguity and that
    every tensor is on q's device, and calls ``attn_fwd`` with that device
    current, on ``stream`` (default: that device's current stream).

    ``check_status=True`` synchronises the stream afterwards and raises
    AttnError if a device-side wait ran out (``attn_sync_status``).  The status
    word behind it is one per device, shared by every stream and caller on that
    device: reading it also clears a timeout that another stream's kernel left.
    """
    import torch
    device = _check_attention_tensors((("q", q), ("k", k), ("v", v), ("out", out), ("lse", lse)))
    B, Hq, S, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or (Bk, Sk, Dk) != (B, S, D):
        raise ValueError("q [B,Hq,S,D] and k, v [B,Hkv,S,D] disagree")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(device):
        if out is None:
            out = torch.empty_like(q)
        if lse is None and return_lse:
            lse = torch.empty((B, Hq, S), dtype=torch.float32, device=device)
        st = _device_stream(device, stream)
        attn_fwd(q, k, v, out, lse, B, Hq, Hkv, S, D, scale, causal, st)
        if check_status:
            attn_sync_status(st)
    return (out, lse) if return_lse else out


def _attention_function():
    """A torch.autograd.Function over the C ABI: forward and backward are the
    library's entry points (argument marshalling only)."""
    import torch

    class AttentionFunction(torch.autograd.Function):
        @staticmethod
        def forward(ctx, q, k, v, causal, scale, block_mask, keep_bits, dropout_p, seed, offset,
                    check_status):
            B, Hq, S, D = q.shape
            Hkv = k.shape[1]
            with torch.cuda.device(q.device):
                out = torch.empty_like(q)
                lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
                opts = options(block_mask=block_mask, keep_bits=keep_bits, dropout_p=dropout_p, seed=seed,
                               offset=offset)
                st = torch.cuda.current_stream(q.device)
                attn_fwd_ex(q, k, v, out, lse, B, Hq, Hkv, S, D, scale, causal, opts, st)
                if check_status:
                    attn_sync_status(st)
            ctx.save_for_backward(q, k, v, out, lse)
            ctx.masks = (block_mask, keep_bits)
            ctx.args = (causal, scale, dropout_p, seed, offset, check_status)
            return out

        @staticmethod
        def backward(ctx, dout):
            q, k, v, out, lse = ctx.saved_tensors
            block_mask, keep_bits = ctx.masks
            causal, scale, dropout_p, seed, offset, check_status = ctx.args
            B, Hq, S, D = q.shape
            Hkv = k.shape[1]
            dout = dout.contiguous()
            _check_attention_tensors((("q", q), ("dout", dout)))
            with torch.cuda.device(q.device):
                dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
                delta = torch.empty_like(lse)
                opts = options(block_mask=block_mask, keep_bits=keep_bits, dropout_p=dropout_p, seed=seed,
                               offset=offset)
                st = torch.cuda.current_stream(q.device)
                attn_bwd_ex(q, k, v, out, dout, lse, delta, dq, dk, dv, B, Hq, Hkv, S, D, scale, causal, opts,
                            st)
                if check_status:
                    attn_sync_status(st)
            return dq, dk, dv, None, None, None, None, None, None, None, None

    return AttentionFunction


_ATTENTION_FUNCTION = None


def attention_trainable(q, k, v, causal: bool = True, scale: float | None = None, block_mask=None,
                        keep_bits=None, dropout_p: float = 0.0, seed: int = 0, offset: int = 0,
                        check_status: bool = False):
    """O = attention(q, k, v) with gradients: forward and backward run the C ABI
    (attn_fwd_ex / attn_bwd_ex with the given options) with q's device current,
    on its current stream.  q [B,Hq,S,D], k/v [B,Hkv,S,D] bf16 CUDA tensors;
    block_mask uint8 [1 or Hq, nt, nt]; keep_bits uint8 [1 or Hq, S, 16*nt];
    dropout combines with either or both.  Every tensor must be on q's device.
    ``check_status=True`` reads the per-device status word after each pass (as
    ``attention`` does) and raises AttnError on a device-side timeout."""
    global _ATTENTION_FUNCTION
    _check_attention_tensors((("q", q), ("k", k), ("v", v), ("block_mask", block_mask),
                              ("keep_bits", keep_bits)))
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    if _ATTENTION_FUNCTION is None:
        _ATTENTION_FUNCTION = _attention_function()
    return _ATTENTION_FUNCTION.apply(q, k, v, bool(causal), float(scale), block_mask, keep_bits,
                                     float(dropout_p), int(seed), int(offset), bool(check_status))
