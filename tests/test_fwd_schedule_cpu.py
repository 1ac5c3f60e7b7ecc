"""The forward kernel's work order (attn_fwd_schedule, host code only): every
unit exactly once, the same assignment as an independent list-scheduling
simulation written here, CTA loads balanced under the cost model, head blocks
taken in turn, and the fall-back cases (table too small) reported."""
import heapq

import pytest

from causal_scaled_dot_gb300 import native
from causal_scaled_dot_gb300.native import ATTN_ERR_INVALID_ARG

HEAD_BLOCK = 16

# (batch_heads, num_q_tiles, causal), all with at least two units per CTA at
# 152 CTAs: the benchmark workloads (B*Hq, S/128), odd tile counts, head counts
# that are not a multiple of the block, fewer heads than a block, non-causal.
SHAPES = [(64, 32, True), (64, 64, True), (64, 32, False), (288, 6, True), (40, 16, True), (35, 17, True),
          (10, 64, True), (37, 33, False), (4096, 2, True)]


def unit_cost(m, nq, causal):
    """Tile products of pair m (query tiles 2m and 2m + 1) plus 2."""
    if not causal:
        return 2 * nq + 2
    return min(2 * m + 1, nq) + min(2 * m + 2, nq) + 2


def simulate(bh_count, nq, causal, ctas):
    """List scheduling restated: units head block by head block, heaviest
    pair first, each to the earliest free CTA (the lower index on ties)."""
    npairs = (nq + 1) // 2
    free = [(0, c) for c in range(ctas)]
    heapq.heapify(free)
    lists = [[] for _ in range(ctas)]
    for b0 in range(0, bh_count, HEAD_BLOCK):
        for m in range(npairs - 1, -1, -1):
            for bh in range(b0, min(b0 + HEAD_BLOCK, bh_count)):
                t, c = heapq.heappop(free)
                lists[c].append((npairs - 1 - m) * bh_count + bh)
                heapq.heappush(free, (t + unit_cost(m, nq, causal), c))
    return lists


@pytest.mark.parametrize("bh_count,nq,causal", SHAPES)
def test_schedule_covers_every_unit_once_and_matches_the_simulation(bh_count, nq, causal):
    npairs = (nq + 1) // 2
    ctas = 152
    lists = native.fwd_schedule(bh_count, nq, causal, ctas)
    assert lists is not None
    flat = [u for lst in lists for u in lst]
    assert sorted(flat) == list(range(bh_count * npairs))
    assert lists == simulate(bh_count, nq, causal, ctas)


@pytest.mark.parametrize("bh_count,nq,causal", [(64, 32, True), (64, 64, True), (64, 32, False), (40, 16, True)])
def test_schedule_balance(bh_count, nq, causal):
    """Max over CTAs of the summed unit cost against the mean: never more than
    one unit above it, and within 2 % at the causal benchmark shapes (equal
    non-causal units split 6 or 7 per CTA whatever the order)."""
    npairs = (nq + 1) // 2
    lists = native.fwd_schedule(bh_count, nq, causal, 152)
    loads = [sum(unit_cost(npairs - 1 - u // bh_count, nq, causal) for u in lst) for lst in lists]
    mean = sum(loads) / len(loads)
    heaviest = max(unit_cost(m, nq, causal) for m in range(npairs))
    assert max(loads) <= mean + heaviest
    if causal and bh_count * npairs >= 4 * 152:
        assert max(loads) <= 1.02 * mean


@pytest.mark.parametrize("bh_count,nq", [(64, 32), (64, 64), (40, 16)])
def test_schedule_takes_head_blocks_in_turn(bh_count, nq):
    """Each CTA's units come block by block: the head block never goes back."""
    lists = native.fwd_schedule(bh_count, nq, True, 152)
    for lst in lists:
        blocks = [(u % bh_count) // HEAD_BLOCK for u in lst]
        assert blocks == sorted(blocks)


def test_schedule_reports_when_the_kernel_keeps_its_arithmetic_order():
    assert native.fwd_schedule(4097, 1, True, 152) is None      # 4097 units: more than the table
    assert native.fwd_schedule(4096, 2, True, 152) is not None   # exactly 4096 units
    assert native.fwd_schedule(64, 32, True, 161) is None        # more CTAs than the table
    assert native.fwd_schedule(64, 32, True, 160) is not None
    assert native.fwd_schedule(32, 16, True, 152) is None        # 256 units: under two per CTA
    assert native.fwd_schedule(38, 16, True, 152) is not None    # 304 units: two per CTA
    assert native.fwd_schedule(37, 16, True, 152) is None        # 296 units


@pytest.mark.parametrize("args", [(0, 32, 1, 152), (64, 0, 1, 152), (64, 32, 1, 0)])
def test_schedule_rejects_bad_sizes(args):
    import ctypes
    import numpy as np
    u16p = ctypes.POINTER(ctypes.c_ushort)
    order = np.zeros(4096, dtype=np.uint16)
    start = np.zeros(161, dtype=np.uint16)
    lib = native.load()
    assert lib.attn_fwd_schedule(*args, order.ctypes.data_as(u16p), start.ctypes.data_as(u16p)) == \
        ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_schedule(64, 32, 1, 152, None, start.ctypes.data_as(u16p)) == ATTN_ERR_INVALID_ARG
