"""The E4M3 rounding model behind the FP8 parity bound (tests/gpu_util.py),
checked on CPU against cases worked by hand."""
import math

import numpy as np
import torch

from tests.gpu_util import fp8_rounding_model


def _codes(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_single_key_rows_are_exact():
    q = _codes(np.ones((1, 1, 1, 16)))
    k = _codes(np.ones((1, 1, 1, 16)))
    v = _codes(np.arange(16, dtype=np.float32).reshape(1, 1, 1, 16))
    assert fp8_rounding_model(q, k, v, (1.0, 1.0, 1.0), 0.25, True) == 0.0


def test_two_keys_by_hand():
    """Row 1 sees keys 0 and 1.  With q = 1 and keys 0 and log2-scores 0 and
    log2(0.3) (scale chosen so), the weights are 0.3 and 1; 0.3 rounds to
    0.3125 in E4M3 (1.25 * 2^-2), 1 is exact.  With v_0 = 1 and v_1 = 0 the
    output moves from 0.3/1.3 to 0.3125/1.3; row 0 (one key) is exact."""
    D = 16
    q = np.zeros((1, 1, 2, D), np.float32)
    q[0, 0, 1, 0] = 1.0
    k = np.zeros((1, 1, 2, D), np.float32)
    k[0, 0, 0, 0] = 1.0
    v = np.zeros((1, 1, 2, D), np.float32)
    v[0, 0, 0, 0] = 1.0
    scale = float(np.float32(math.log(0.3)))  # score of key 0 for row 1: log(0.3) nats
    got = fp8_rounding_model(_codes(q), _codes(k), _codes(v), (1.0, 1.0, 1.0), scale, True, rows=[1])
    w0 = math.exp(float(np.float32(scale)))  # the model's exact weight (0.3 to float32 precision)
    want = abs(0.3125 - w0) / w0
    assert abs(got - want) < 1e-9, (got, want)
