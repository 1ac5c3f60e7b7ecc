"""GPU parity when the persistent forward kernel runs more than one round of
units per CTA: units of even rounds walk their key tiles upwards, units of odd
rounds downwards with their two query tiles swapped.  Small sizes with more
units than a GB300 has SMs (B2 H48 S700: 288 units for 152 CTAs) put units
into both directions; every row is compared with the fp64 oracle, for each
variant of the kernel (bf16 at D = 64 and 128, causal and not, block masks,
element masks with and without a block mask, dropout, E4M3 inputs), and the
block-masked and element-masked kernels with masks that keep everything must
reproduce the unmasked call bit for bit, also in the descending units."""
import math

import numpy as np
import pytest

import oracle
from causal_scaled_dot_gb300.inputs import (block_mask_of_keep_bits, qkv_bf16, qkv_e4m3,
                                            random_block_mask, random_keep_bits, window_keep_bits)
from tests.gpu_util import (compare, compare_fp8, compare_masked, fp8_rounding_model, run_gpu, run_gpu_dropout,
                            run_gpu_elem_masked, run_gpu_fp8, run_gpu_masked)

pytestmark = pytest.mark.gpu

B, HQ, HKV, S = 2, 48, 12, 700  # 3 query-tile pairs per head: 288 units


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    units = B * HQ * ((S + 127) // 128 + 1) // 2
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert units > sms, "the shape must give more units than CTAs"


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_two_rounds_plain(D, causal):
    q, k, v = qkv_bf16(B, HQ, HKV, S, D, seed=7100 + D)
    scale = 1.0 / math.sqrt(D)
    o, l, _ = run_gpu(q, k, v, scale, causal)
    o_ref, l_ref = oracle.attention(q, k, v, scale, causal)
    print(compare(o, o_ref, l, l_ref, f"two rounds D{D} causal={causal}"))


@pytest.mark.parametrize("causal", [True, False])
def test_two_rounds_block_mask(causal):
    D = 128
    q, k, v = qkv_bf16(B, HQ, HKV, S, D, seed=7200)
    scale = 1.0 / math.sqrt(D)
    mask = random_block_mask(HQ, S, 0.6, seed=72)
    o, l = run_gpu_masked(q, k, v, scale, causal, mask)
    o_ref, l_ref = oracle.attention_masked(q, k, v, scale, mask, causal)
    print(compare_masked(o, o_ref, l, l_ref, f"two rounds block mask causal={causal}"))


@pytest.mark.parametrize("with_block_mask", [False, True])
def test_two_rounds_elem_mask(with_block_mask):
    D = 64
    q, k, v = qkv_bf16(B, HQ, HKV, S, D, seed=7300)
    scale = 1.0 / math.sqrt(D)
    bits = window_keep_bits(S, 200) & random_keep_bits(1, S, 0.8, seed=73)
    bm = block_mask_of_keep_bits(bits, S) if with_block_mask else None
    o, l = run_gpu_elem_masked(q, k, v, scale, True, bits, bm)
    o_ref, l_ref = oracle.attention_keep(q, k, v, scale, bits, True, block_mask=bm)
    print(compare_masked(o, o_ref, l, l_ref, f"two rounds elem mask block={with_block_mask}"))


def test_two_rounds_dropout():
    D, p = 128, 0.2
    q, k, v = qkv_bf16(B, HQ, HKV, S, D, seed=7400)
    scale = 1.0 / math.sqrt(D)
    p8 = int(round(p * 256))
    o, l = run_gpu_dropout(q, k, v, scale, True, p, 0xABC, 3)
    o_ref, l_ref = oracle.attention_dropout(q, k, v, scale, p8, 0xABC, 3, True)
    print(compare(o, o_ref, l, l_ref, "two rounds dropout", abs_scale=256.0 / (256 - p8)))


def test_two_rounds_e4m3():
    D = 128
    q, k, v = qkv_e4m3(B, HQ, HKV, S, D, seed=7500)
    descales = (1.0, 1.0, 1.0)
    scale = 1.0 / math.sqrt(D)
    o, l = run_gpu_fp8(q, k, v, descales, scale, True)
    o_ref, l_ref = oracle.attention_e4m3(q, k, v, scale, descales, True)
    model = fp8_rounding_model(q, k, v, descales, scale, True)
    print(compare_fp8(o, o_ref, l, l_ref, oracle.e4m3_decode(v), "two rounds e4m3", model_rel=model))


@pytest.mark.parametrize("causal", [True, False])
def test_two_rounds_all_keeping_masks_equal_unmasked_bitwise(causal):
    D = 128
    q, k, v = qkv_bf16(B, HQ, HKV, S, D, seed=7600)
    scale = 1.0 / math.sqrt(D)
    nt = (S + 127) // 128
    o_u, l_u, _ = run_gpu(q, k, v, scale, causal)
    o_m, l_m = run_gpu_masked(q, k, v, scale, causal, np.ones((1, nt, nt), np.uint8))
    assert np.array_equal(o_m, o_u) and np.array_equal(l_m, l_u)
    ones = np.full((1, S, 16 * nt), 0xFF, np.uint8)
    o_e, l_e = run_gpu_elem_masked(q, k, v, scale, causal, ones)
    assert np.array_equal(o_e, o_u) and np.array_equal(l_e, l_u)
