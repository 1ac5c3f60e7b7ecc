// fwd_schedule.h -- the order in which the persistent forward kernel's CTAs
// take their work units, computed on the host once per shape.
//
// A unit is (flat head bh = b*Hq + hq, query-tile pair m: tiles 2m and 2m+1),
// numbered u = (npairs - 1 - m) * BH + bh as decode_unit (kernel_ws.cuh)
// reads it.  Causal units differ in size (a pair needs key tiles up to its
// diagonal), so the order must balance the CTAs; and every unit of a head
// reads that head's K and V, so the CTAs running at one time should share few
// heads: then the K/V tiles they read are still in L2 when the next unit of
// the same head asks for them.
//
// The builder hands the units out head block by head block (kHeadBlock query
// heads at a time, all their pairs, heaviest pair first within the block),
// each unit to the CTA that frees up first under a cost model of its tile
// products -- list scheduling, whose result depends only on the shape and the
// CTA count, so the kernel's results stay deterministic.  A block of 16 heads
// at S = 4096 holds 32 MB of K and V, well inside L2; a least-recently-used
// model of L2 gives no K/V re-reads at B4 H16 S4096 or B2 H32 S8192 with this
// order, against 1.29x and 3.8x the K/V bytes with the arithmetic
// boustrophedon order, at the same balance (max/mean CTA cost 1.014).
//
// With fewer than two units per CTA the kernel keeps its arithmetic order:
// there every CTA runs one or two units, the boustrophedon pairs the heaviest
// with the lightest, and the K/V of all heads fit in L2 anyway (B1 H32 S2048,
// 256 units: 38.0 us against 38.7 us with the table; B4 H16 S4096, 1024 units:
// 198.8 us against 202.5 us, DRAM reads 361 -> 201 MB).
//
// Header-only and free of CUDA calls, so host tests can compile it alone.
#pragma once

#include <cstdint>
#include <functional>
#include <algorithm>
#include <vector>

namespace attn {
namespace host {

constexpr int kHeadBlock = 16;

// Cost of unit pair m in tile products (one QK^T and one PV per key tile of
// each query tile) plus a fixed 2 for the unit's start and end.
inline long long fwd_unit_cost(int m, int nq, bool causal) {
    if (!causal) return 2LL * nq + 2;
    const int n0 = 2 * m + 1 < nq ? 2 * m + 1 : nq;
    const int n1 = 2 * m + 2 < nq ? 2 * m + 2 : nq;
    return (long long)n0 + n1 + 2;
}

// Whether the kernel takes its units from a table for this many units and CTAs.
inline bool fwd_schedule_wanted(long long units, int grid) { return units >= 2LL * grid; }

// Fills start[0 .. grid] and order[0 .. units): CTA c runs order[start[c]] ..
// order[start[c + 1] - 1].  Returns false (and writes nothing) when the units
// or CTAs exceed the capacities given or an argument is out of range.
inline bool build_fwd_schedule(int bh_count, int nq, bool causal, int grid, int max_units, int max_ctas,
                               uint16_t* start, uint16_t* order) {
    if (bh_count <= 0 || nq <= 0 || grid <= 0 || grid > max_ctas) return false;
    const long long npairs = (nq + 1) / 2;
    const long long units = (long long)bh_count * npairs;
    if (units > max_units || units > 65535) return false;
    // Pass 1: the CTA of each unit in hand-out order, from a min-heap of
    // (time the CTA frees up) << 8 | CTA: the earliest first, ties to the lower CTA.
    std::vector<uint16_t> unit_of((size_t)units), cta_of((size_t)units);
    std::vector<uint64_t> heap;
    heap.reserve((size_t)grid);
    for (int c = 0; c < grid; ++c) heap.push_back((uint64_t)c);  // already a valid min-heap
    const auto later = std::greater<uint64_t>();
    size_t k = 0;
    for (int b0 = 0; b0 < bh_count; b0 += kHeadBlock) {
        const int b1 = b0 + kHeadBlock < bh_count ? b0 + kHeadBlock : bh_count;
        for (long long m = npairs - 1; m >= 0; --m) {
            const uint64_t cost = (uint64_t)fwd_unit_cost((int)m, nq, causal) << 8;
            for (int bh = b0; bh < b1; ++bh, ++k) {
                std::pop_heap(heap.begin(), heap.end(), later);
                unit_of[k] = (uint16_t)((npairs - 1 - m) * bh_count + bh);
                cta_of[k] = (uint16_t)(heap.back() & 0xFFu);
                heap.back() += cost;
                std::push_heap(heap.begin(), heap.end(), later);
            }
        }
    }
    // Pass 2: group by CTA, keeping each CTA's units in hand-out order.
    std::vector<int> fill((size_t)grid + 1, 0);
    for (size_t i = 0; i < k; ++i) ++fill[(size_t)cta_of[i] + 1];
    for (int c = 0; c < grid; ++c) fill[(size_t)c + 1] += fill[(size_t)c];
    for (int c = 0; c <= grid; ++c) start[c] = (uint16_t)fill[(size_t)c];
    for (size_t i = 0; i < k; ++i) order[fill[cta_of[i]]++] = unit_of[i];
    return true;
}

}  // namespace host
}  // namespace attn
