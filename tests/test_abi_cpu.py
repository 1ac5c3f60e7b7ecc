"""The C-ABI library builds, loads and exports every declared symbol; argument
errors are reported before any device work (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from causal_scaled_dot_gb300 import native
from causal_scaled_dot_gb300.native import (ATTN_ERR_INVALID_ARG, ATTN_ERR_MISALIGNED,
                                            ATTN_ERR_UNSUPPORTED)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(attn_\w+)\s*\(", text, flags=re.M)
    return names


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("attn_fwd", "attn_fwd_fp8", "attn_fwd_block_masked", "attn_fwd_elem_masked",
                     "attn_fwd_dropout",
                     "attn_bwd", "attn_bwd_block_masked", "attn_out_proj", "attn_status_string",
                     "attn_sync_status"):
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = native.load()
    for name in declared_functions():
        assert hasattr(lib, name), f"libattn.so does not export {name}"
    out = subprocess.run(["nm", "-D", "--defined-only", native.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\b(attn_\w+)\b", out))
    assert set(declared_functions()) <= exported


def test_status_strings_and_version():
    for code in range(7):
        assert native.attn_status_string(code).startswith("ATTN_")
    assert "unknown" in native.attn_status_string(99)
    assert native.attn_version() >= 100


def _call(q=16, k=32, v=48, out=64, lse=None, B=1, Hq=2, Hkv=2, S=128, D=128, scale=0.1,
          causal=1):
    lib = native.load()
    return lib.attn_fwd(q, k, v, out, lse, B, Hq, Hkv, S, D, ctypes.c_float(scale), causal, None)


# Fake, never-dereferenced pointer values far apart so they do not overlap.
P = dict(q=1 << 40, k=2 << 40, v=3 << 40, out=4 << 40)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), ATTN_ERR_INVALID_ARG),
    (dict(k=None), ATTN_ERR_INVALID_ARG),
    (dict(v=None), ATTN_ERR_INVALID_ARG),
    (dict(out=None), ATTN_ERR_INVALID_ARG),
    (dict(B=0), ATTN_ERR_INVALID_ARG),
    (dict(Hq=0), ATTN_ERR_INVALID_ARG),
    (dict(Hkv=0), ATTN_ERR_INVALID_ARG),
    (dict(S=0), ATTN_ERR_INVALID_ARG),
    (dict(S=-5), ATTN_ERR_INVALID_ARG),
    (dict(Hq=6, Hkv=4), ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), ATTN_ERR_INVALID_ARG),
    (dict(scale=-0.1), ATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), ATTN_ERR_INVALID_ARG),
    (dict(D=96), ATTN_ERR_UNSUPPORTED),
    (dict(D=256), ATTN_ERR_UNSUPPORTED),
    (dict(q=(1 << 40) + 8), ATTN_ERR_MISALIGNED),
    (dict(out=(4 << 40) + 2), ATTN_ERR_MISALIGNED),
    (dict(lse=(5 << 40) + 2), ATTN_ERR_MISALIGNED),
    (dict(out=1 << 40), ATTN_ERR_INVALID_ARG),            # out aliases q
    (dict(out=(2 << 40) + 4096), ATTN_ERR_INVALID_ARG),   # out overlaps k
    (dict(lse=(4 << 40) + 1024), ATTN_ERR_INVALID_ARG),   # lse overlaps out
])
def test_argument_errors_are_rejected_before_launch(kw, code):
    args = dict(P)
    args.update(kw)
    assert _call(**args) == code


def test_python_binding_rejects_host_tensors():
    import torch
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        native.attn_fwd(q, q, q, q, None, 1, 1, 1, 8, 64, 0.125, True, stream=0)
    with pytest.raises(ValueError):
        native.attention(q, q, q)
    with pytest.raises(ValueError, match="CUDA"):
        native.attention_trainable(q, q, q)
    with pytest.raises(ValueError, match="bf16"):
        native.attention_trainable(q.float(), q, q)


class _FakeCudaTensor:
    """Stands in for a bf16 CUDA tensor on a given device (no GPU needed)."""

    def __init__(self, index, shape=(1, 2, 128, 64)):
        import torch
        self.is_cuda = True
        self.dtype = torch.bfloat16
        self.device = torch.device("cuda", index)
        self.shape = shape

    def dim(self):
        return len(self.shape)

    def is_contiguous(self):
        return True


def test_python_wrappers_reject_tensors_on_different_devices(monkeypatch):
    """The C ABI runs on the calling thread's current device: tensors split over
    two devices are refused before the library is loaded or called."""
    def no_library():
        raise AssertionError("the library must not be reached")

    monkeypatch.setattr(native, "load", no_library)
    a, b = _FakeCudaTensor(0), _FakeCudaTensor(1)
    for args in ((a, b, a), (a, a, b), (b, a, a)):
        with pytest.raises(ValueError, match="same device"):
            native.attention(*args)
        with pytest.raises(ValueError, match="same device"):
            native.attention_trainable(*args)
    with pytest.raises(ValueError, match="same device"):
        native.attention(a, a, a, out=b)
    with pytest.raises(ValueError, match="same device"):
        native.attention_trainable(a, a, a, block_mask=b)


def test_selftest_rejects_bad_limits():
    lib = native.load()
    assert lib.attn_selftest_wait_timeout(0, None) == ATTN_ERR_INVALID_ARG
    assert lib.attn_selftest_wait_timeout(2000000, None) == ATTN_ERR_INVALID_ARG


def _call_fp8(q=1 << 40, k=2 << 40, v=3 << 40, out=4 << 40, lse=None, dq=1.0, dk=1.0, dv=1.0, B=1,
              Hq=2, Hkv=2, S=128, D=128, scale=0.1, causal=1):
    lib = native.load()
    f = ctypes.c_float
    return lib.attn_fwd_fp8(q, k, v, f(dq), f(dk), f(dv), out, lse, B, Hq, Hkv, S, D, f(scale),
                            causal, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), ATTN_ERR_INVALID_ARG),
    (dict(dq=0.0), ATTN_ERR_INVALID_ARG),
    (dict(dk=-1.0), ATTN_ERR_INVALID_ARG),
    (dict(dv=float("nan")), ATTN_ERR_INVALID_ARG),
    (dict(D=64), ATTN_ERR_UNSUPPORTED),
    (dict(Hq=3, Hkv=2), ATTN_ERR_INVALID_ARG),
    (dict(k=(2 << 40) + 4), ATTN_ERR_MISALIGNED),
    (dict(out=(1 << 40) + 64), ATTN_ERR_INVALID_ARG),  # out overlaps q
])
def test_fp8_argument_errors_are_rejected_before_launch(kw, code):
    assert _call_fp8(**kw) == code


def _call_masked(mask=5 << 40, mask_heads=1, q=1 << 40, k=2 << 40, v=3 << 40, out=4 << 40,
                 lse=None, B=1, Hq=2, Hkv=2, S=300, D=128, scale=0.1, causal=1):
    lib = native.load()
    return lib.attn_fwd_block_masked(q, k, v, out, lse, B, Hq, Hkv, S, D, ctypes.c_float(scale),
                                     causal, mask, mask_heads, None)


@pytest.mark.parametrize("kw,code", [
    (dict(mask=None), ATTN_ERR_INVALID_ARG),
    (dict(mask_heads=0), ATTN_ERR_INVALID_ARG),
    (dict(mask_heads=3), ATTN_ERR_INVALID_ARG),   # neither 1 nor Hq
    (dict(mask_heads=-2), ATTN_ERR_INVALID_ARG),
    (dict(q=None), ATTN_ERR_INVALID_ARG),
    (dict(Hq=3, Hkv=2, mask_heads=3), ATTN_ERR_INVALID_ARG),
    (dict(D=96), ATTN_ERR_UNSUPPORTED),
    (dict(v=(3 << 40) + 2), ATTN_ERR_MISALIGNED),
])
def test_masked_argument_errors_are_rejected_before_launch(kw, code):
    assert _call_masked(**kw) == code


def _call_elem(keep=6 << 40, keep_heads=1, mask=None, mask_heads=1, q=1 << 40, k=2 << 40,
               v=3 << 40, out=4 << 40, lse=None, B=1, Hq=2, Hkv=2, S=300, D=128, scale=0.1,
               causal=1):
    lib = native.load()
    return lib.attn_fwd_elem_masked(q, k, v, out, lse, B, Hq, Hkv, S, D, ctypes.c_float(scale),
                                    causal, keep, keep_heads, mask, mask_heads, None)


@pytest.mark.parametrize("kw,code", [
    (dict(keep=None), ATTN_ERR_INVALID_ARG),
    (dict(keep_heads=0), ATTN_ERR_INVALID_ARG),
    (dict(keep_heads=3), ATTN_ERR_INVALID_ARG),   # neither 1 nor Hq
    (dict(mask=5 << 40, mask_heads=3), ATTN_ERR_INVALID_ARG),
    (dict(keep=(6 << 40) + 8), ATTN_ERR_MISALIGNED),
    (dict(q=None), ATTN_ERR_INVALID_ARG),
    (dict(D=96), ATTN_ERR_UNSUPPORTED),
    (dict(k=(2 << 40) + 2), ATTN_ERR_MISALIGNED),
])
def test_elem_masked_argument_errors_are_rejected_before_launch(kw, code):
    assert _call_elem(**kw) == code


def test_elem_masked_bwd_rejects_bad_masks_before_launch():
    lib = native.load()
    args = [1 << 40, 2 << 40, 3 << 40, 4 << 40, 5 << 40, 6 << 40, 7 << 40, 8 << 40, 9 << 40,
            10 << 40, 1, 2, 2, 300, 128, ctypes.c_float(0.1), 1]
    ok_bits = 11 << 40
    assert lib.attn_bwd_elem_masked(*args, None, 1, None, 1, None) == ATTN_ERR_INVALID_ARG
    assert lib.attn_bwd_elem_masked(*args, ok_bits, 3, None, 1, None) == ATTN_ERR_INVALID_ARG
    assert lib.attn_bwd_elem_masked(*args, ok_bits, 1, 12 << 40, 3, None) == ATTN_ERR_INVALID_ARG
    assert lib.attn_bwd_elem_masked(*args, ok_bits + 4, 1, None, 1, None) == ATTN_ERR_MISALIGNED
    assert lib.attn_bwd_elem_masked(*args[:14], 96, *args[15:], ok_bits, 1, None, 1, None) == ATTN_ERR_UNSUPPORTED


def test_dropout_bwd_rejects_bad_rates_before_launch():
    lib = native.load()
    args = [1 << 40, 2 << 40, 3 << 40, 4 << 40, 5 << 40, 6 << 40, 7 << 40, 8 << 40, 9 << 40,
            10 << 40, 1, 2, 2, 300, 128, ctypes.c_float(0.1), 1]
    for bad in (-0.1, float("nan"), float("inf"), 0.999):
        assert lib.attn_bwd_dropout(*args, ctypes.c_float(bad), 1, 2, None) == ATTN_ERR_INVALID_ARG
    assert lib.attn_bwd_dropout(*args[:14], 96, *args[15:], ctypes.c_float(0.1), 1, 2, None) == ATTN_ERR_UNSUPPORTED


def test_masks_overlapping_outputs_are_rejected_before_launch():
    """A block mask or keep bits that overlap O / LSE (forward) or dQ / dK / dV /
    delta (backward) is an argument error."""
    lib = native.load()
    q, k, v, out = 1 << 40, 2 << 40, 3 << 40, 4 << 40
    B, Hq, Hkv, S, D = 1, 2, 2, 300, 128
    f = ctypes.c_float(0.1)
    # forward: a block mask inside O, keep bits inside LSE
    assert lib.attn_fwd_block_masked(q, k, v, out, None, B, Hq, Hkv, S, D, f, 1, out + 4096, 1,
                                     None) == ATTN_ERR_INVALID_ARG
    lse = 5 << 40
    assert lib.attn_fwd_elem_masked(q, k, v, out, lse, B, Hq, Hkv, S, D, f, 1, lse + 1024, 1, None, 1,
                                    None) == ATTN_ERR_INVALID_ARG
    # backward: keep bits inside dK
    bargs = [q, k, v, out, 6 << 40, lse, 7 << 40, 8 << 40, 9 << 40, 10 << 40, B, Hq, Hkv, S, D, f, 1]
    assert lib.attn_bwd_elem_masked(*bargs, (9 << 40) + 4096, 1, None, 1, None) == ATTN_ERR_INVALID_ARG
    assert lib.attn_bwd_block_masked(*bargs, (7 << 40) + 64, 1, None) == ATTN_ERR_INVALID_ARG


def test_options_struct_layout_matches_the_header(tmp_path):
    """attn_options_t as gcc lays it out from include/attn.h equals the binding's ctypes
    structure, field by field."""
    fields = [f for f, _ in native.AttnOptions._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "attn.h"\nint main(void) {\n'
                   '  printf("%zu\\n", sizeof(attn_options_t));\n'
                   + "".join(f'  printf("%zu\\n", offsetof(attn_options_t, {f}));\n' for f in fields)
                   + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    want = [ctypes.sizeof(native.AttnOptions)] + [getattr(native.AttnOptions, f).offset for f in fields]
    assert got == want


def test_unsupported_option_combinations_are_rejected_before_launch():
    lib = native.load()
    q, k, v, out = 1 << 40, 2 << 40, 3 << 40, 4 << 40
    f = ctypes.c_float(0.1)
    fp8_drop = native.options(e4m3_descales=(1.0, 1.0, 1.0), dropout_p=0.1)
    assert lib.attn_fwd_ex(q, k, v, out, None, 1, 2, 2, 300, 128, f, 1, ctypes.byref(fp8_drop),
                           None) == ATTN_ERR_UNSUPPORTED
    fp8_d64 = native.options(e4m3_descales=(1.0, 1.0, 1.0))
    assert lib.attn_fwd_ex(q, k, v, out, None, 1, 2, 2, 300, 64, f, 1, ctypes.byref(fp8_d64),
                           None) == ATTN_ERR_UNSUPPORTED
    bad_fmt = native.options()
    bad_fmt.input_format = 7
    assert lib.attn_fwd_ex(q, k, v, out, None, 1, 2, 2, 300, 128, f, 1, ctypes.byref(bad_fmt),
                           None) == ATTN_ERR_INVALID_ARG
    bargs = [q, k, v, out, 6 << 40, 5 << 40, 7 << 40, 8 << 40, 9 << 40, 10 << 40, 1, 2, 2, 300, 128, f, 1]
    assert lib.attn_bwd_ex(*bargs, ctypes.byref(fp8_d64), None) == ATTN_ERR_UNSUPPORTED


def test_keep_bit_packing():
    from causal_scaled_dot_gb300.inputs import (block_mask_of_keep_bits, keep_row_bytes, pack_keep_bits,
                                                random_keep_bits, unpack_keep_bits, window_keep_bits)
    assert keep_row_bytes(1) == 16 and keep_row_bytes(128) == 16 and keep_row_bytes(129) == 32
    b = random_keep_bits(2, 300, 0.4, seed=3)
    assert b.shape == (2, 300, 48) and np.array_equal(b, random_keep_bits(2, 300, 0.4, seed=3))
    keep = unpack_keep_bits(b, 300)
    assert abs(float(keep.mean()) - 0.4) < 0.01
    assert np.array_equal(pack_keep_bits(keep), b)
    # bit j % 8 of byte j / 8, padding bits zero
    one = np.zeros((1, 130, 130), bool)
    one[0, 5, 129] = True
    packed = pack_keep_bits(one)
    assert packed[0, 5, 16] == 2 and packed.sum() == 2
    w = unpack_keep_bits(window_keep_bits(300, 64), 300)[0]
    i, j = np.nonzero(w)
    assert np.all((j <= i) & (j > i - 64)) and w.sum() == sum(min(64, r + 1) for r in range(300))
    bm = block_mask_of_keep_bits(window_keep_bits(600, 100), 600)[0]
    assert bm.shape == (5, 5) and np.array_equal(bm, np.eye(5, dtype=np.uint8) + np.eye(5, k=-1, dtype=np.uint8))


def test_random_block_mask_shape_and_density():
    from causal_scaled_dot_gb300.inputs import random_block_mask
    m = random_block_mask(4, 1000, 0.3, seed=9)
    assert m.shape == (4, 8, 8) and m.dtype == np.uint8
    assert set(np.unique(m)) <= {0, 1}
    assert np.array_equal(m, random_block_mask(4, 1000, 0.3, seed=9))
    big = random_block_mask(1, 128 * 200, 0.3, seed=1)
    assert abs(float(big.mean()) - 0.3) < 0.01
    assert random_block_mask(1, 256, 0.0, seed=1).sum() == 0
    assert random_block_mask(1, 256, 1.0, seed=1).all()


def _call_bwd(q=1 << 40, k=2 << 40, v=3 << 40, out=4 << 40, dout=5 << 40, lse=6 << 40,
              delta=7 << 40, dq=8 << 40, dk=9 << 40, dv=10 << 40, B=1, Hq=2, Hkv=2, S=300, D=128,
              scale=0.1, causal=1):
    lib = native.load()
    return lib.attn_bwd(q, k, v, out, dout, lse, delta, dq, dk, dv, B, Hq, Hkv, S, D,
                        ctypes.c_float(scale), causal, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), ATTN_ERR_INVALID_ARG),
    (dict(dout=None), ATTN_ERR_INVALID_ARG),
    (dict(lse=None), ATTN_ERR_INVALID_ARG),
    (dict(delta=None), ATTN_ERR_INVALID_ARG),
    (dict(dv=None), ATTN_ERR_INVALID_ARG),
    (dict(S=0), ATTN_ERR_INVALID_ARG),
    (dict(Hq=3, Hkv=2), ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), ATTN_ERR_INVALID_ARG),
    (dict(D=96), ATTN_ERR_UNSUPPORTED),
    (dict(dout=(5 << 40) + 8), ATTN_ERR_MISALIGNED),
    (dict(dk=(9 << 40) + 2), ATTN_ERR_MISALIGNED),
    (dict(delta=(7 << 40) + 2), ATTN_ERR_MISALIGNED),
    (dict(dq=(1 << 40) + 4096), ATTN_ERR_INVALID_ARG),      # dq overlaps q
    (dict(dk=(8 << 40) + 4096), ATTN_ERR_INVALID_ARG),      # dk overlaps dq
    (dict(delta=(10 << 40) + 64), ATTN_ERR_INVALID_ARG),    # delta overlaps dv
    (dict(dv=(6 << 40)), ATTN_ERR_INVALID_ARG),             # dv overlaps lse
])
def test_bwd_argument_errors_are_rejected_before_launch(kw, code):
    assert _call_bwd(**kw) == code


def _call_dropout(p=0.1, q=1 << 40, k=2 << 40, v=3 << 40, out=4 << 40, lse=None, B=1, Hq=2, Hkv=2,
                  S=300, D=128, scale=0.1, causal=1):
    lib = native.load()
    return lib.attn_fwd_dropout(q, k, v, out, lse, B, Hq, Hkv, S, D, ctypes.c_float(scale), causal,
                                ctypes.c_float(p), 1, 2, None)


@pytest.mark.parametrize("kw,code", [
    (dict(p=-0.01), ATTN_ERR_INVALID_ARG),
    (dict(p=1.0), ATTN_ERR_INVALID_ARG),          # rounds to p8 = 256
    (dict(p=0.999), ATTN_ERR_INVALID_ARG),        # rounds to p8 = 256
    (dict(p=float("nan")), ATTN_ERR_INVALID_ARG),
    (dict(p=float("inf")), ATTN_ERR_INVALID_ARG),
    (dict(q=None), ATTN_ERR_INVALID_ARG),
    (dict(D=80), ATTN_ERR_UNSUPPORTED),
    (dict(k=(2 << 40) + 8), ATTN_ERR_MISALIGNED),
])
def test_dropout_argument_errors_are_rejected_before_launch(kw, code):
    assert _call_dropout(**kw) == code


def test_dropout_offsets_past_32_bits_are_rejected_before_launch():
    """The offset is the fourth 32-bit counter word of the generator: 2^32 and
    above are argument errors in every dropout entry point (with dropout on);
    without dropout the offset is not used."""
    lib = native.load()
    q, k, v, out = 1 << 40, 2 << 40, 3 << 40, 4 << 40
    f = ctypes.c_float(0.1)
    big = 1 << 32
    assert lib.attn_fwd_dropout(q, k, v, out, None, 1, 2, 2, 300, 128, f, 1, f, 1, big, None) == ATTN_ERR_INVALID_ARG
    bargs = [q, k, v, out, 6 << 40, 5 << 40, 7 << 40, 8 << 40, 9 << 40, 10 << 40, 1, 2, 2, 300, 128, f, 1]
    assert lib.attn_bwd_dropout(*bargs, f, 1, big, None) == ATTN_ERR_INVALID_ARG
    drop = native.options(dropout_p=0.1, seed=1, offset=big)
    assert lib.attn_fwd_ex(q, k, v, out, None, 1, 2, 2, 300, 128, f, 1, ctypes.byref(drop), None) == ATTN_ERR_INVALID_ARG
    assert lib.attn_bwd_ex(*bargs, ctypes.byref(drop), None) == ATTN_ERR_INVALID_ARG
    # the largest offset passes the argument checks (and then fails only for want of a device here)
    assert lib.attn_fwd_dropout(q, k, v, out, None, 1, 2, 2, 300, 128, f, 1, f, 1, big - 1, None) != ATTN_ERR_INVALID_ARG


def _call_proj(out=1 << 40, w=2 << 40, bias=None, y=3 << 40, B=1, H=4, S=300, D=128, E=512):
    lib = native.load()
    return lib.attn_out_proj(out, w, bias, y, B, H, S, D, E, None)


@pytest.mark.parametrize("kw,code", [
    (dict(out=None), ATTN_ERR_INVALID_ARG),
    (dict(w=None), ATTN_ERR_INVALID_ARG),
    (dict(y=None), ATTN_ERR_INVALID_ARG),
    (dict(E=0), ATTN_ERR_INVALID_ARG),
    (dict(S=0), ATTN_ERR_INVALID_ARG),
    (dict(E=12), ATTN_ERR_UNSUPPORTED),
    (dict(D=32), ATTN_ERR_UNSUPPORTED),
    (dict(w=(2 << 40) + 8), ATTN_ERR_MISALIGNED),
    (dict(bias=(4 << 40) + 2), ATTN_ERR_MISALIGNED),
    (dict(y=(1 << 40) + 4096), ATTN_ERR_INVALID_ARG),   # y overlaps out
    (dict(y=(2 << 40)), ATTN_ERR_INVALID_ARG),          # y is w
])
def test_proj_argument_errors_are_rejected_before_launch(kw, code):
    assert _call_proj(**kw) == code


def test_masked_bwd_rejects_bad_masks_before_launch():
    lib = native.load()
    args = [1 << 40, 2 << 40, 3 << 40, 4 << 40, 5 << 40, 6 << 40, 7 << 40, 8 << 40, 9 << 40, 10 << 40,
            1, 2, 2, 300, 128, ctypes.c_float(0.1), 1]
    assert lib.attn_bwd_block_masked(*args, None, 1, None) == ATTN_ERR_INVALID_ARG
    assert lib.attn_bwd_block_masked(*args, 11 << 40, 3, None) == ATTN_ERR_INVALID_ARG
    assert lib.attn_bwd_block_masked(*args[:14], 96, *args[15:], 11 << 40, 1, None) == ATTN_ERR_UNSUPPORTED


def _size_cases():
    """(name, call, tensors) per Python wrapper: host tensors of exactly the sizes
    that B=1, Hq=4, Hkv=2, S=130, D=64 (E=64) imply."""
    import torch
    B, Hq, Hkv, S, D, E = 1, 4, 2, 130, 64, 64
    nt = 2
    bf, u8, f32 = torch.bfloat16, torch.uint8, torch.float32
    qs, kvs = (B, Hq, S, D), (B, Hkv, S, D)

    def fwd(in_dtype=bf):
        return dict(q=torch.zeros(qs, dtype=in_dtype), k=torch.zeros(kvs, dtype=in_dtype),
                    v=torch.zeros(kvs, dtype=in_dtype), out=torch.zeros(qs, dtype=bf),
                    lse=torch.zeros((B, Hq, S), dtype=f32))

    def bwd():
        t = fwd()
        t.update(dout=torch.zeros(qs, dtype=bf), delta=torch.zeros((B, Hq, S), dtype=f32),
                 dq=torch.zeros(qs, dtype=bf), dk=torch.zeros(kvs, dtype=bf), dv=torch.zeros(kvs, dtype=bf))
        return t

    bm = lambda: torch.zeros((Hq, nt, nt), dtype=u8)  # noqa: E731
    kb = lambda: torch.zeros((1, S, 16 * nt), dtype=u8)  # noqa: E731
    dims = (B, Hq, Hkv, S, D, 0.125, True)
    F = ("q", "k", "v", "out", "lse")
    G = ("q", "k", "v", "out", "dout", "lse", "delta", "dq", "dk", "dv")

    def opts_with(t):
        o = native.options()
        o.tensors = (t.get("block_mask"), t.get("keep_bits"))
        if "block_mask" in t:
            o.block_mask, o.mask_heads = t["block_mask"].data_ptr(), Hq
        if "keep_bits" in t:
            o.keep_bits, o.keep_heads = t["keep_bits"].data_ptr(), 1
        return o

    cases = [
        ("attn_fwd", lambda t: native.attn_fwd(*(t[n] for n in F), *dims, stream=0), fwd()),
        ("attn_fwd_fp8", lambda t: native.attn_fwd_fp8(t["q"], t["k"], t["v"], 1.0, 1.0, 1.0, t["out"], t["lse"],
                                                       *dims, stream=0), fwd(u8)),
        ("attn_fwd_block_masked", lambda t: native.attn_fwd_block_masked(*(t[n] for n in F), *dims,
                                                                         t["block_mask"], Hq, stream=0),
         dict(fwd(), block_mask=bm())),
        ("attn_fwd_elem_masked", lambda t: native.attn_fwd_elem_masked(*(t[n] for n in F), *dims, t["keep_bits"], 1,
                                                                       t["block_mask"], Hq, stream=0),
         dict(fwd(), keep_bits=kb(), block_mask=bm())),
        ("attn_fwd_dropout", lambda t: native.attn_fwd_dropout(*(t[n] for n in F), *dims, 0.1, 1, 2, stream=0),
         fwd()),
        ("attn_fwd_ex", lambda t: native.attn_fwd_ex(*(t[n] for n in F), *dims, opts_with(t), stream=0),
         dict(fwd(), keep_bits=kb(), block_mask=bm())),
        ("attn_bwd", lambda t: native.attn_bwd(*(t[n] for n in G), *dims, stream=0), bwd()),
        ("attn_bwd_block_masked", lambda t: native.attn_bwd_block_masked(*(t[n] for n in G), *dims,
                                                                         t["block_mask"], Hq, stream=0),
         dict(bwd(), block_mask=bm())),
        ("attn_bwd_elem_masked", lambda t: native.attn_bwd_elem_masked(*(t[n] for n in G), *dims, t["keep_bits"], 1,
                                                                       t["block_mask"], Hq, stream=0),
         dict(bwd(), keep_bits=kb(), block_mask=bm())),
        ("attn_bwd_dropout", lambda t: native.attn_bwd_dropout(*(t[n] for n in G), *dims, 0.1, 1, 2, stream=0),
         bwd()),
        ("attn_bwd_ex", lambda t: native.attn_bwd_ex(*(t[n] for n in G), *dims, opts_with(t), stream=0),
         dict(bwd(), keep_bits=kb(), block_mask=bm())),
        ("attn_out_proj", lambda t: native.attn_out_proj(t["out"], t["w"], t["bias"], t["y"], B, Hq, S, D, E,
                                                         stream=0),
         dict(out=torch.zeros(qs, dtype=bf), w=torch.zeros((E, Hq * D), dtype=bf), bias=torch.zeros(E, dtype=f32),
              y=torch.zeros((B, S, E), dtype=bf))),
    ]
    return cases


@pytest.mark.parametrize("case", range(12), ids=lambda i: _size_cases()[i][0])
def test_python_binding_checks_tensor_sizes(case):
    """Every wrapper checks, before it passes an address on, that each tensor
    holds the bytes its sizes imply (the C entry points cannot): exactly sized
    host tensors pass that check and are then refused as host memory; any one
    argument one element short is refused by name as too small."""
    name, call, tensors = _size_cases()[case]
    with pytest.raises(ValueError, match="CUDA device memory"):
        call(tensors)
    for arg in tensors:
        short = dict(tensors)
        short[arg] = tensors[arg].reshape(-1)[:-1].clone()
        with pytest.raises(ValueError, match=f"^{arg} holds"):
            call(short)


def test_binding_fails_loudly_without_its_library(monkeypatch):
    """With no library loaded and none that can be built, every entry point
    raises: there is no other path to fall back on."""
    def no_build(*args, **kwargs):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libattn")

    monkeypatch.setattr(native, "_lib", None)
    monkeypatch.setattr(native._build, "build", no_build)
    with pytest.raises(RuntimeError, match="nvcc"):
        native.load()
    with pytest.raises(RuntimeError, match="nvcc"):
        native.attn_version()
    with pytest.raises(RuntimeError, match="nvcc"):
        native.attn_fwd(None, None, None, None, None, 1, 1, 1, 8, 64, 0.125, True, stream=0)


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "attn.h"

int main(void) {
    attn_options_t o;
    if (attn_version() < 100) return 1;
    if (strncmp(attn_status_string(ATTN_ERR_MISALIGNED), "ATTN_", 5) != 0) return 2;
    /* argument errors return before any device work */
    if (attn_fwd(NULL, NULL, NULL, NULL, NULL, 1, 1, 1, 8, 64, 0.125f, 1, NULL) != ATTN_ERR_INVALID_ARG)
        return 3;
    memset(&o, 0, sizeof o);
    o.input_format = 7;
    if (attn_fwd_ex(NULL, NULL, NULL, NULL, NULL, 1, 1, 1, 8, 64, 0.125f, 1, &o, NULL) != ATTN_ERR_INVALID_ARG)
        return 4;
    if (attn_bwd(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 1, 1, 1, 8, 64, 0.125f, 1,
                 NULL) != ATTN_ERR_INVALID_ARG)
        return 5;
    puts("ok");
    return 0;
}
"""


def test_plain_c_program_links_and_calls_the_library(tmp_path):
    """A C99 program that includes only attn.h and links libattn.so: the entry
    points have C linkage and the header's signatures resolve; calls that return
    before any device work give their documented codes."""
    lib_dir = os.path.dirname(native.library_path())
    native.load()  # built and current
    src = tmp_path / "use_attn.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "use_attn"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                    "-L", lib_dir, "-lattn", f"-Wl,-rpath,{lib_dir}", "-o", str(exe)], check=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert res.returncode == 0 and res.stdout.strip() == "ok", (res.returncode, res.stdout, res.stderr)
