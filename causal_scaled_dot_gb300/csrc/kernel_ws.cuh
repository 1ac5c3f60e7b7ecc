// kernel_ws.cuh -- warp-specialised, persistent attention forward for sm_103a.
//
// Work unit: one (batch, query head) and a pair of adjacent 128-row query
// tiles (2m, 2m+1).  Units are numbered heaviest causal pairs first (pair
// index descending), query heads that share a key/value head next to each
// other.  One CTA per SM takes its units in the order of a table the host
// computes per shape (fwd_schedule.h: head block by head block, so that the
// K/V tiles of the heads in flight stay in L2, each unit to the CTA that
// frees up first), or, without a table, in boustrophedon rounds -- round r
// gives unit r*G + c to CTA c on even rounds and to CTA G-1-c on odd ones --
// which balances the sorted unit costs with no global state either way.
//
// Roles (384 threads, 12 warps):
//   warp 0      TMA producer: Q tiles of the unit, then K_j, V_j into a ring
//               of single-tile shared-memory slots.
//   warp 1      MMA issuer (one thread) and TMEM owner: S_i = Q_i K_j^T
//               (both operands in shared memory) and O_i += P_i V_j (P read
//               from tensor memory).
//   warps 2-3   idle (a separate correction warpgroup measured slower).
//   warps 4-7   softmax warpgroup 0: one thread per row of query tile 2m.
//   warps 8-11  softmax warpgroup 1: one thread per row of query tile 2m+1.
// The two warpgroups ping-pong: while one runs its softmax the tensor core
// computes the other's products.  At the end of a unit each softmax warp also
// drains its 32 rows of O (tensor memory -> x 1/l -> bf16 -> a shared-memory
// box -> TMA store) and writes their LSE.  The drain of query tile 2m
// overlaps the tensor core's last products for tile 2m+1; a separate
// correction warpgroup for the drain (16 warps) measured slower.
//
// Tensor memory (512 columns x 128 lanes, fp32): S_0 [0,128), S_1 [128,256),
// O_0 [256, 256+D), O_1 [256+D, 256+2D).  P_i (bf16, two per column) is written
// over the upper half of S_i, columns [64,128) of it, after S_i has been read.
//
// Online softmax: the running maximum m (in log2 units, scale*log2(e)*s) is
// raised only when a tile's maximum exceeds it by more than kRescaleSlack;
// otherwise probabilities up to 2^kRescaleSlack are kept against the stale
// m.  O and l are always relative to the same m, so the final O / l and
// LSE = (m + log2 l) ln 2 are unaffected; O is rescaled in TMEM only when m
// actually moves.  When S_i(j) is observed complete, every earlier MMA of the
// issuing thread -- in particular O_i += P_i(j-1) V_{j-1} -- has completed
// too (tcgen05.commit tracks all prior operations), so the softmax thread may
// rescale O_i then without a further barrier.
//
// The steps are those of the naive causal attention in the "Profiling in
// PyTorch (Part 3)" retelling (section "Naive Attention": QK^T, scale,
// causal -inf mask, softmax, times V), fused with the tiled online softmax
// that the same retelling describes for FlashAttention-2 ("The Flash
// Backend"); key tiles entirely after a query tile are never loaded, and
// only diagonal tiles are masked.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "philox.cuh"
#include "ptx.cuh"

namespace attn {

constexpr float kRescaleSlack = 8.0f;  // log2 units: probabilities stay <= 256

// F selects FP8 E4M3 inputs (one byte per element; D = 128 only, so that a
// 128-byte swizzle row is one 128-element row of a tile); otherwise bf16.
template <int D, bool F>
struct WsLayout {
    static_assert(!F || D == 128, "FP8 inputs need D = 128");
    static constexpr int kElemBytes = F ? 1 : 2;
    static constexpr int kRowElems = 128 / kElemBytes;       // elements per 128-byte row
    static constexpr int kThreads = 384;
    // Registers per thread after the split: warps 0-3 (producer, MMA issuer,
    // idle) shrink, the softmax warps grow.  Launch allocation: 384 x 168 =
    // 64512 = 128 x kRegsSmall + 256 x kRegsSoftmax.
    static constexpr int kRegsSmall = 72;
    static constexpr int kRegsSoftmax = 216;
    static_assert(128 * kRegsSmall + 256 * kRegsSoftmax <= kThreads * 168, "register split");
    static constexpr uint32_t kTileBytes = kTile * D * kElemBytes;  // 32 KB at bf16 D = 128
    static constexpr int kStages = (kTileBytes == 32768) ? 4 : 8;    // K/V ring slots, one tile each
    static constexpr int kChunks = D / kRowElems;                    // 128-byte swizzle blocks
    static constexpr uint32_t kChunkBytes = kTile * 128;   // one block of a tile: 16 KB
    // Output staging: per softmax warp, 32 rows x 64 columns of O as bf16 in
    // the 128-byte swizzled layout of the O tensor map's {64 columns, 32 rows}
    // box (4 KB), filled and stored once per 64-column block.
    static constexpr uint32_t kOutBoxBytes = 32 * 128;
    static constexpr uint32_t kQ0 = 0;
    static constexpr uint32_t kQ1 = kTileBytes;
    static constexpr uint32_t kRing = 2 * kTileBytes;
    static constexpr uint32_t kStage = kRing + kStages * kTileBytes;
    static constexpr uint32_t kBars = kStage + 8 * kOutBoxBytes;
    // mbarrier indices
    static constexpr int kQFull = 0, kQEmpty = 2, kSFull = 4, kPFull = 6, kOFull = 8;
    static constexpr int kKVFull = 10, kKVEmpty = 10 + kStages, kDrain = 10 + 2 * kStages;
    static constexpr int kOEmpty = kDrain + 1;  // block-masked kernels: O_i read out (2 barriers)
    static constexpr int kNumBars = kDrain + 3;
    static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kBytes = kAbort + 4;
    static constexpr uint32_t kDynamicSmem = kBytes + 1024;  // slack for 1024-byte alignment
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kDynamicSmem <= 227 * 1024, "shared memory budget");
    static_assert(kStage % 1024 == 0, "staging boxes need the swizzle atom's alignment");
};

// Unit u -> (bh, pair m).  Causal: heaviest pairs first.  Within a pair index
// consecutive u walk bh = b*Hq + hq, so GQA siblings are adjacent.  n0 / n1
// bound the key tiles of the unit's query tiles qt[0] / qt[1] (causality,
// sequence end); with a block mask some tiles below the bound are dropped too
// (tile_active).
//
// Key direction: units of odd rounds walk their key tiles from the highest
// down to 0, and units of even rounds from 0 up.  The
// CTAs of one round run their units roughly in step, so a round ends on the
// key tiles the next round starts with and those are still in L2 (a
// least-recently-used model of the profile shape, B4 H16 S4096, puts the
// K/V bytes read from DRAM at 273 MB instead of 471 MB).  A descending unit
// swaps its query tiles -- qt[0] = 2m+1, qt[1] = 2m -- so that query tile 0
// always holds the key tile the other lacks at the unit's boundary with the
// previous unit: first in a descending unit, last in an ascending one (the
// issuer starts a unit's first S_0 inside the previous unit).  The order is
// fixed by the unit's round, so results are deterministic for a given grid.
struct Unit {
    int bh, hq, m, kv_bh, n0, n1, n;
    int qt[2];  // query tiles of softmax warpgroups 0 and 1
    bool desc;  // key tiles visited from n-1 down to 0
};
__device__ __forceinline__ Unit decode_unit(int u, const FwdParams& p, bool desc = false) {
    const int BH = p.B * p.Hq;
    const int npairs = (p.num_q_tiles + 1) >> 1;
    Unit w;
    w.m = npairs - 1 - u / BH;
    w.bh = u - (u / BH) * BH;
    const int b = w.bh / p.Hq;
    const int hq = w.bh - b * p.Hq;
    w.hq = hq;
    w.kv_bh = b * p.Hkv + hq / p.group;
    w.desc = desc;
    w.qt[0] = 2 * w.m + (desc ? 1 : 0);
    w.qt[1] = 2 * w.m + (desc ? 0 : 1);
    if (p.causal) {
        w.n0 = min(w.qt[0] + 1, p.num_q_tiles);
        w.n1 = min(w.qt[1] + 1, p.num_q_tiles);
    } else {
        w.n0 = w.n1 = p.num_q_tiles;
    }
    w.n = max(w.n0, w.n1);
    return w;
}
// The key direction of the units of round r.
__device__ __forceinline__ bool round_desc(int r) { return (r & 1) != 0; }
// Key tile visited at step s (0 <= s < n) of a unit without a block mask.
__device__ __forceinline__ int key_of_step(const Unit& w, int s) { return w.desc ? w.n - 1 - s : s; }

// Does query tile qt[i] of unit w use key tile j?  M (block mask present) is
// a template flag so that the unmasked kernel keeps its plain counting loops:
// without a mask, tile i uses key tiles [0, n_i) (the odd last query tile of a
// pair, past the sequence end, runs too and writes nothing).  With a mask, a
// tile below n_i is used when the mask keeps it, and a query tile past the
// sequence end uses none.
template <bool M>
__device__ __forceinline__ bool tile_active(const FwdParams& p, const Unit& w, int i, int j) {
    if (j >= (i == 0 ? w.n0 : w.n1)) return false;
    if constexpr (!M) {
        return true;
    } else {
        const int qt = w.qt[i];
        if (qt >= p.num_q_tiles) return false;
        const int nt = p.num_q_tiles;
        return __ldg(p.block_mask + ((size_t)(p.mask_heads == 1 ? 0 : w.hq) * nt + qt) * nt + j) != 0;
    }
}
// Visit order of a unit's key tiles with a block mask: the union of both query
// tiles' kept tiles, ascending or descending with the unit.  -1 ends the walk.
template <bool M>
__device__ __forceinline__ int next_visit(const FwdParams& p, const Unit& w, int j) {
    if (w.desc) {
        for (--j; j >= 0; --j)
            if (tile_active<M>(p, w, 0, j) || tile_active<M>(p, w, 1, j)) return j;
    } else {
        for (++j; j < w.n; ++j)
            if (tile_active<M>(p, w, 0, j) || tile_active<M>(p, w, 1, j)) return j;
    }
    return -1;
}
template <bool M>
__device__ __forceinline__ int first_visit(const FwdParams& p, const Unit& w) {
    return next_visit<M>(p, w, w.desc ? w.n : -1);
}
// The key tile query tile i uses last in the unit's visit order (-1 if none).
template <bool M>
__device__ __forceinline__ int last_visit(const FwdParams& p, const Unit& w, int i) {
    const int n_i = i == 0 ? w.n0 : w.n1;
    if (w.desc) {
        for (int j = 0; j < n_i; ++j)
            if (tile_active<M>(p, w, i, j)) return j;
    } else {
        for (int j = n_i - 1; j >= 0; --j)
            if (tile_active<M>(p, w, i, j)) return j;
    }
    return -1;
}

// The unit this CTA runs in round r (>= num_units: no more work): from the
// host's table when it has one, else the boustrophedon order -- round r
// takes units [rG, rG + G), even rounds by CTA index, odd rounds in reverse,
// so that with units sorted heaviest first a CTA's heavy unit of one round
// pairs with a light one of the next.
__device__ __forceinline__ int unit_of_round(const FwdSchedule& sc, int num_units, int r) {
    const int c = blockIdx.x;
    if (sc.enabled) {
        const int i = (int)sc.start[c] + r;
        return i < (int)sc.start[c + 1] ? (int)sc.order[i] : num_units;
    }
    const int G = gridDim.x;
    return r * G + ((r & 1) ? (G - 1 - c) : c);
}

template <int D, bool F>
__device__ __forceinline__ uint32_t ws_bar(uint32_t base, int i) {
    return base + WsLayout<D, F>::kBars + 8u * (uint32_t)i;
}

// ---------------------------------------------------------------- producer
template <int D, bool F, bool M, bool DR, bool E>
__device__ void ws_load_role(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                             const CUtensorMap* tm_v, const FwdParams& p, const FwdSchedule& sc, uint32_t base,
                             volatile int* abort_flag) {
    using L = WsLayout<D, F>;
    uint32_t qe_phase[2] = {0u, 0u};
    int slot = 0;
    uint32_t ring_phase = 0;
    // Loads issued and possibly not yet landed, for the drain after an abort.
    uint32_t pend_kv = 0, pend_kv_par = 0, pend_q = 0, pend_q_par = 0;
    const uint64_t lim = p.wait_limit_ns;
    // Q is read once per unit: its lines leave L2 first, which keeps room for
    // the K/V tiles that the other query tiles of the head read again (ncu:
    // DRAM reads 399 -> 370 MB per launch at B4 H16 S4096 D128, with the O
    // stores marked the same way).
    const uint64_t read_once = ptx::policy_evict_first();
    // Q_i of a unit into its slot once the previous unit's last S_i = Q_i K^T
    // has completed.
    auto load_q = [&](const Unit& w, int i) -> bool {
        if (!ptx::mbar_wait(ws_bar<D, F>(base, L::kQEmpty + i), qe_phase[i] ^ 1u, abort_flag, p.status, lim))
            return false;
        qe_phase[i] ^= 1u;
        const uint32_t full = ws_bar<D, F>(base, L::kQFull + i);
        ptx::mbar_arrive_expect_tx(full, L::kTileBytes);
        const uint32_t dst = base + (i == 0 ? L::kQ0 : L::kQ1);
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c)
            ptx::tma_load_3d_hint(dst + c * L::kChunkBytes, tm_q, full, c * L::kRowElems, w.qt[i] * kTile, w.bh,
                                  read_once);
        pend_q |= 1u << i;
        pend_q_par = (pend_q_par & ~(1u << i)) | (((qe_phase[i] ^ 1u) & 1u) << i);
        return true;
    };
    for (int rnd = 0, u = unit_of_round(sc, p.num_units, 0); u < p.num_units;
             u = unit_of_round(sc, p.num_units, ++rnd)) {
        const Unit w = decode_unit(u, p, round_desc(rnd));
        // Without a block mask the issuer starts a unit's first S_0 = Q_0 K_0^T
        // while the previous unit's last softmax runs (see the MMA role), so
        // the unit's first K is loaded right after Q_0: Q_1's slot frees only
        // with the previous unit's last S_1, and K_0 need not wait for it.
        bool q1_loaded = false;
        if (!load_q(w, 0)) goto drain;
        if (M) {
            if (!load_q(w, 1)) goto drain;
            q1_loaded = true;
        }
        // Key tiles in the order the issuer consumes them: every step of the
        // unit's direction without a block mask, the union of both query
        // tiles' kept tiles in that direction with one.
        for (int st = 0, j = M ? first_visit<M>(p, w) : key_of_step(w, 0); M ? j >= 0 : st < w.n;
             ++st, j = M ? next_visit<M>(p, w, j) : key_of_step(w, st)) {
#pragma unroll
            for (int t = 0; t < 2; ++t) {  // t = 0: K_j, t = 1: V_j
                if (!ptx::mbar_wait(ws_bar<D, F>(base, L::kKVEmpty + slot), ring_phase ^ 1u, abort_flag,
                                    p.status, lim))
                    goto drain;
                const uint32_t full = ws_bar<D, F>(base, L::kKVFull + slot);
                ptx::mbar_arrive_expect_tx(full, L::kTileBytes);
                const uint32_t dst = base + L::kRing + (uint32_t)slot * L::kTileBytes;
                const CUtensorMap* map = t == 0 ? tm_k : tm_v;
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c)
                    ptx::tma_load_3d(dst + c * L::kChunkBytes, map, full, c * L::kRowElems, j * kTile, w.kv_bh);
                pend_kv |= 1u << slot;
                pend_kv_par = (pend_kv_par & ~(1u << slot)) | (ring_phase << slot);
                if (++slot == L::kStages) {
                    slot = 0;
                    ring_phase ^= 1u;
                }
                if (!q1_loaded) {
                    if (!load_q(w, 1)) goto drain;
                    q1_loaded = true;
                }
            }
        }
        if (!q1_loaded && !load_q(w, 1)) goto drain;
    }
    return;
drain:
    // Let every copy already issued land before the CTA can exit.
    for (int s = 0; s < L::kStages; ++s)
        if (pend_kv & (1u << s))
            ptx::drain_wait(ws_bar<D, F>(base, L::kKVFull + s), (pend_kv_par >> s) & 1u, lim);
    for (int i = 0; i < 2; ++i)
        if (pend_q & (1u << i))
            ptx::drain_wait(ws_bar<D, F>(base, L::kQFull + i), ((pend_q_par >> i) & 1u) ^ 0u, lim);
}

// ---------------------------------------------------------------- MMA issuer
// The issuing thread spins on its barriers (mbar_wait_spin): it alone feeds
// the tensor core, which idles while it waits, so it should see a completed
// phase at once (+0.8 % at B4 H16 S4096 D128 against suspend-hinted waits);
// the other roles keep the suspend hint, so that their waiting warps leave
// issue slots to the softmax warps on their schedulers.
template <int D, bool F, bool M, bool DR, bool E>
__device__ void ws_mma_role(const FwdParams& p, const FwdSchedule& sc, uint32_t base, uint32_t tmem,
                            volatile int* abort_flag) {
    using L = WsLayout<D, F>;
    constexpr uint32_t kIdescS = F ? ptx::idesc_e4m3_f32(kTile, kTile, false)
                                   : ptx::idesc_bf16_f32(kTile, kTile, false);
    constexpr uint32_t kIdescO = F ? ptx::idesc_e4m3_f32(kTile, D, true)
                                   : ptx::idesc_bf16_f32(kTile, D, true);
    const uint64_t lim = p.wait_limit_ns;
    uint32_t qf_phase = 0;
    uint32_t pf_phase[2] = {0u, 0u};
    int slot = 0;
    uint32_t ring_phase = 0;

    // S_i = Q_i K^T with K in ring slot `ks`: all K steps from one asm block.
    auto issue_s = [&](int i, int ks) {
        const uint64_t a = ptx::sdesc_sw128(base + (i == 0 ? L::kQ0 : L::kQ1), 16, 1024);
        const uint64_t b = ptx::sdesc_sw128(base + L::kRing + (uint32_t)ks * L::kTileBytes, 16, 1024);
        if constexpr (F)
            ptx::mma_ss_f8_k128(tmem + (uint32_t)i * kTile, a, b, kIdescS, 0u);
        else if constexpr (D == 128)
            ptx::mma_ss_k128(tmem + (uint32_t)i * kTile, a, b, kIdescS, 0u);
        else
            ptx::mma_ss_k64(tmem + (uint32_t)i * kTile, a, b, kIdescS, 0u);
        ptx::mma_commit(ws_bar<D, F>(base, L::kSFull + i));
    };
    // O_i (+)= P_i V with V in slot `vs`.  bf16: P_i in TMEM columns [64,128) of
    // S_i, keys 0-63 then keys 64-127 (8 KB further into V, 32 TMEM columns
    // further into P).  FP8: P_i in columns [96,128), all 128 keys at once.
    auto issue_pv = [&](int i, int vs, bool accumulate) {
        const uint64_t v = ptx::sdesc_sw128(base + L::kRing + (uint32_t)vs * L::kTileBytes,
                                            L::kChunkBytes, 1024);
        const uint32_t o = tmem + 256u + (uint32_t)i * D;
        if constexpr (F) {
            ptx::mma_ts_f8_k128(o, tmem + (uint32_t)i * kTile + 96u, v, kIdescO, accumulate ? 1u : 0u);
        } else {
            const uint32_t pcol = tmem + (uint32_t)i * kTile + 64u;
            ptx::mma_ts_k64(o, pcol, v, kIdescO, accumulate ? 1u : 0u);
            ptx::mma_ts_k64(o, pcol + 32u, v + 512u, kIdescO, 1u);
        }
    };
    auto wait_ring = [&](int& got) -> bool {
        if (!ptx::mbar_wait_spin(ws_bar<D, F>(base, L::kKVFull + slot), ring_phase, abort_flag, p.status, lim))
            return false;
        got = slot;
        if (++slot == L::kStages) {
            slot = 0;
            ring_phase ^= 1u;
        }
        ptx::tc_fence_after();
        return true;
    };
    auto wait_p = [&](int i) -> bool {
        if (!ptx::mbar_wait_spin(ws_bar<D, F>(base, L::kPFull + i), pf_phase[i], abort_flag, p.status, lim))
            return false;
        pf_phase[i] ^= 1u;
        ptx::tc_fence_after();
        return true;
    };
    // Block-masked kernels: a query tile without key tiles makes no P handshake,
    // so before O_i of a unit is produced (or declared empty) the previous
    // unit's O_i must have been read out -- otherwise OFull_i could run two
    // phases ahead of the softmax warps waiting on it.  Once per tile per unit.
    uint32_t oe_phase[2] = {1u, 1u};
    auto wait_o_empty = [&](int i) -> bool {
        if (!ptx::mbar_wait_spin(ws_bar<D, F>(base, L::kOEmpty + i), oe_phase[i], abort_flag, p.status, lim))
            return false;
        oe_phase[i] ^= 1u;
        ptx::tc_fence_after();
        return true;
    };

    if constexpr (!M) {
        // Without a block mask both query tiles use every key tile below their
        // causal bound.  In a unit's last step the issuer starts the next
        // unit's first product S_0 = Q_0 K^T before the final O_1 += P_1 V,
        // whose P_1 the other softmax warpgroup is still computing: otherwise
        // the tensor core idles through that softmax and again through the
        // next unit's first one.  S_0's tensor memory is free (P_0 has been
        // consumed) and the softmax warps of tile 0 publish the next P_0 only
        // after reading O_0 out, so O_0 is not overwritten early.
        bool pre = false;  // this unit's first S_0 was issued during the previous unit
        int pre_kslot = 0;
        for (int rnd = 0, u = unit_of_round(sc, p.num_units, 0); u < p.num_units;
             u = unit_of_round(sc, p.num_units, ++rnd)) {
            const Unit w = decode_unit(u, p, round_desc(rnd));
            if (!pre && !ptx::mbar_wait_spin(ws_bar<D, F>(base, L::kQFull + 0), qf_phase, abort_flag, p.status, lim))
                break;
            ptx::tc_fence_after();
            // Step s visits key tile key_of_step(w, s); query tile i uses it when
            // that key tile is below n_i.  Ascending: tile i uses steps
            // [0, n_i); descending: steps [n - n_i, n).  Tile 0 uses step 0
            // either way (n0 >= n1 when descending).
            const int n = w.n;
            const int first1 = w.desc ? n - w.n1 : 0;
            const int last0 = w.desc ? n - 1 : w.n0 - 1, last1 = w.desc ? n - 1 : w.n1 - 1;
            auto act0 = [&](int st) { return w.desc || st < w.n0; };
            auto act1 = [&](int st) { return st >= first1 && st <= last1; };
            int kslot, vslot;
            if (pre) {
                kslot = pre_kslot;
            } else {
                if (!wait_ring(kslot)) break;
                issue_s(0, kslot);
                if (last0 == 0) ptx::mma_commit(ws_bar<D, F>(base, L::kQEmpty + 0));
            }
            pre = false;
            // Q_1 is waited for only now: at the kernel's start S_0 need not wait
            // for Q_1's copy too.
            if (!ptx::mbar_wait_spin(ws_bar<D, F>(base, L::kQFull + 1), qf_phase, abort_flag, p.status, lim)) break;
            qf_phase ^= 1u;
            ptx::tc_fence_after();
            if (act1(0)) {
                issue_s(1, kslot);
                if (last1 == 0) ptx::mma_commit(ws_bar<D, F>(base, L::kQEmpty + 1));
            }
            ptx::mma_commit(ws_bar<D, F>(base, L::kKVEmpty + kslot));
            bool ok = true;
            for (int st = 0; st < n; ++st) {
                const int sn = st + 1;
                if (!(ok = wait_ring(vslot))) break;
                if (act0(st)) {
                    if (!(ok = wait_p(0))) break;
                    issue_pv(0, vslot, st > 0);
                    if (st == last0) ptx::mma_commit(ws_bar<D, F>(base, L::kOFull + 0));
                }
                const bool more = sn < n;
                if (more) {
                    if (!(ok = wait_ring(kslot))) break;
                    if (act0(sn)) {
                        issue_s(0, kslot);
                        if (sn == last0) ptx::mma_commit(ws_bar<D, F>(base, L::kQEmpty + 0));
                    }
                } else {
                    const int u2 = unit_of_round(sc, p.num_units, rnd + 1);
                    if (u2 < p.num_units) {  // the next unit's first S_0
                        const Unit w2 = decode_unit(u2, p, round_desc(rnd + 1));
                        if (!(ok = ptx::mbar_wait_spin(ws_bar<D, F>(base, L::kQFull + 0), qf_phase, abort_flag,
                                                  p.status, lim)))
                            break;
                        ptx::tc_fence_after();
                        if (!(ok = wait_ring(pre_kslot))) break;
                        issue_s(0, pre_kslot);
                        if ((w2.desc ? w2.n : w2.n0) == 1) ptx::mma_commit(ws_bar<D, F>(base, L::kQEmpty + 0));
                        pre = true;
                    }
                }
                if (act1(st)) {
                    if (!(ok = wait_p(1))) break;
                    issue_pv(1, vslot, st > first1);
                    if (st == last1) ptx::mma_commit(ws_bar<D, F>(base, L::kOFull + 1));
                }
                ptx::mma_commit(ws_bar<D, F>(base, L::kKVEmpty + vslot));
                if (more) {
                    if (act1(sn)) {
                        issue_s(1, kslot);
                        if (sn == last1) ptx::mma_commit(ws_bar<D, F>(base, L::kQEmpty + 1));
                    }
                    ptx::mma_commit(ws_bar<D, F>(base, L::kKVEmpty + kslot));
                }
            }
            if (!ok) break;
        }
    } else {
        for (int rnd = 0, u = unit_of_round(sc, p.num_units, 0); u < p.num_units;
             u = unit_of_round(sc, p.num_units, ++rnd)) {
            const Unit w = decode_unit(u, p, round_desc(rnd));
            if (!ptx::mbar_wait_spin(ws_bar<D, F>(base, L::kQFull + 0), qf_phase, abort_flag, p.status, lim) ||
                !ptx::mbar_wait_spin(ws_bar<D, F>(base, L::kQFull + 1), qf_phase, abort_flag, p.status, lim))
                break;
            qf_phase ^= 1u;
            // Key tiles run over the union of both query tiles' active tiles; each
            // product is issued only for a query tile that uses the key tile.
            const int last0 = last_visit<M>(p, w, 0), last1 = last_visit<M>(p, w, 1);
            if (last0 < 0) ptx::mma_commit(ws_bar<D, F>(base, L::kQEmpty + 0));
            if (last1 < 0) ptx::mma_commit(ws_bar<D, F>(base, L::kQEmpty + 1));
            bool first0 = true, first1 = true, ok = true;
            int j = first_visit<M>(p, w);
            int kslot, vslot;
            if (j >= 0) {
                if (!wait_ring(kslot)) break;
                if (tile_active<M>(p, w, 0, j)) {
                    issue_s(0, kslot);
                    if (j == last0) ptx::mma_commit(ws_bar<D, F>(base, L::kQEmpty + 0));
                }
                if (tile_active<M>(p, w, 1, j)) {
                    issue_s(1, kslot);
                    if (j == last1) ptx::mma_commit(ws_bar<D, F>(base, L::kQEmpty + 1));
                }
                ptx::mma_commit(ws_bar<D, F>(base, L::kKVEmpty + kslot));
            }
            while (j >= 0) {
                const int jn = next_visit<M>(p, w, j);
                if (!(ok = wait_ring(vslot))) break;
                if (tile_active<M>(p, w, 0, j)) {
                    if (!(ok = wait_p(0))) break;
                    if (M && first0 && !(ok = wait_o_empty(0))) break;
                    issue_pv(0, vslot, !first0);
                    first0 = false;
                    if (j == last0) ptx::mma_commit(ws_bar<D, F>(base, L::kOFull + 0));
                }
                const bool more = jn >= 0;
                if (more) {
                    if (!(ok = wait_ring(kslot))) break;
                    if (tile_active<M>(p, w, 0, jn)) {
                        issue_s(0, kslot);
                        if (jn == last0) ptx::mma_commit(ws_bar<D, F>(base, L::kQEmpty + 0));
                    }
                }
                if (tile_active<M>(p, w, 1, j)) {
                    if (!(ok = wait_p(1))) break;
                    if (M && first1 && !(ok = wait_o_empty(1))) break;
                    issue_pv(1, vslot, !first1);
                    first1 = false;
                    if (j == last1) ptx::mma_commit(ws_bar<D, F>(base, L::kOFull + 1));
                }
                ptx::mma_commit(ws_bar<D, F>(base, L::kKVEmpty + vslot));
                if (more) {
                    if (tile_active<M>(p, w, 1, jn)) {
                        issue_s(1, kslot);
                        if (jn == last1) ptx::mma_commit(ws_bar<D, F>(base, L::kQEmpty + 1));
                    }
                    ptx::mma_commit(ws_bar<D, F>(base, L::kKVEmpty + kslot));
                }
                j = jn;
            }
            if (!ok) break;
            // A query tile with no key tile still completes its O phase.
            if (last0 < 0) {
                if (!wait_o_empty(0)) break;
                ptx::mma_commit(ws_bar<D, F>(base, L::kOFull + 0));
            }
            if (last1 < 0) {
                if (!wait_o_empty(1)) break;
                ptx::mma_commit(ws_bar<D, F>(base, L::kOFull + 1));
            }
        }
    }
    // Every MMA issued above completes before TMEM can be released.
    ptx::mma_commit(ws_bar<D, F>(base, L::kDrain));
    ptx::drain_wait(ws_bar<D, F>(base, L::kDrain), 0u, lim);
}

// ---------------------------------------------------------------- softmax
template <int D, bool F, bool M, bool DR, bool E>
__device__ void ws_softmax_role(const CUtensorMap* tm_o, const FwdParams& p, const FwdSchedule& sc, uint32_t base,
                                uint32_t tmem, int wg, volatile int* abort_flag) {
    using L = WsLayout<D, F>;
    const int r = threadIdx.x - (4 + 4 * wg) * 32;  // row within the query tile, 0..127
    const int warp_in_wg = r >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t stage = base + L::kStage + (uint32_t)(4 * wg + warp_in_wg) * L::kOutBoxBytes;
    const uint64_t written_once = ptx::policy_evict_first();  // O: no reader in this kernel
    const uint32_t lane_off = (uint32_t)(warp_in_wg * 32) << 16;
    const uint32_t tS = tmem + lane_off + (uint32_t)wg * kTile;
    const uint32_t tP = tS + 64u;
    const uint32_t tO = tmem + lane_off + 256u + (uint32_t)wg * D;
    const uint32_t bar_s = ws_bar<D, F>(base, L::kSFull + wg);
    const uint32_t bar_p = ws_bar<D, F>(base, L::kPFull + wg);
    const uint32_t bar_o = ws_bar<D, F>(base, L::kOFull + wg);
    const float sl2 = p.scale_log2;
    const uint64_t lim = p.wait_limit_ns;
    uint32_t s_phase = 0, o_phase = 0;

    for (int rnd = 0, u = unit_of_round(sc, p.num_units, 0); u < p.num_units;
             u = unit_of_round(sc, p.num_units, ++rnd)) {
        const Unit w = decode_unit(u, p, round_desc(rnd));
        const int qt = w.qt[wg];
        const int n_i = wg == 0 ? w.n0 : w.n1;
        float m_run = 0.f;  // reference maximum (log2 units), set by the first tile
        float l_run = 0.f;
        bool first = true;  // no visible key yet
        // Element-masked kernels: this row's 16 keep bytes per key tile, read
        // one key tile ahead so that the load is not on the tile's critical path.
        const uint8_t* keep_row = nullptr;
        uint4 keep_next = make_uint4(~0u, ~0u, ~0u, ~0u);
        int keep_next_j = -1;
        if constexpr (E) {
            const int row = qt * kTile + r;
            if (row < p.S)
                keep_row = p.keep_bits +
                           ((size_t)(p.keep_heads == 1 ? 0 : w.hq) * p.S + row) * (size_t)p.keep_row_bytes;
        }
        for (int t = 0; t < n_i; ++t) {
            const int j = w.desc ? n_i - 1 - t : t;  // the unit's key direction
            if (!tile_active<M>(p, w, wg, j)) continue;
            uint4 keep = make_uint4(~0u, ~0u, ~0u, ~0u);
            if constexpr (E) {
                if (keep_row != nullptr) {
                    keep = keep_next_j == j ? keep_next : __ldg(reinterpret_cast<const uint4*>(keep_row + 16 * j));
                    if (t + 1 < n_i) {
                        const int jn = w.desc ? j - 1 : j + 1;
                        keep_next = __ldg(reinterpret_cast<const uint4*>(keep_row + 16 * jn));
                        keep_next_j = jn;
                    }
                }
            }
            // Dropout: this tile's keep decisions, made while the warpgroup
            // waits for its scores (the tensor core is still on the other
            // query tile's products): one Philox4x32-10 block per 16 keys of
            // the row, kept as carry-test words (bit 7 of byte b: key
            // 16 blk + 4 w + b is kept).
            uint32_t gw[DR ? 32 : 1];
            if constexpr (DR) {
                const uint32_t c4 = (256u - (uint32_t)p.dropout_p8) * 0x01010101u;
                const uint32_t qrow = (uint32_t)(qt * kTile + r);
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    uint32_t rnd[4];
                    philox4x32_10((uint32_t)(j * 8 + b), qrow, (uint32_t)w.bh, (uint32_t)p.dropout_offset,
                                  p.philox_round_keys, rnd);
#pragma unroll
                    for (int k = 0; k < 4; ++k) gw[4 * b + k] = bytes_ge(rnd[k], c4);
                }
            }
            bool ok = ptx::mbar_wait(bar_s, s_phase, abort_flag, p.status, lim);
            if (!__all_sync(0xffffffffu, ok)) return;
            s_phase ^= 1u;
            ptx::tc_fence_after();

            uint32_t sr[128];
#pragma unroll
            for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tS + c * 32, sr + c * 32);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 4; ++c) ptx::reg_fence32(sr + c * 32);
            float s[128];
#pragma unroll
            for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);

            const int kv0 = j * kTile;
            if (p.causal && j == qt) {
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c > r) s[c] = -INFINITY;  // key after the query
            } else if (!p.causal && kv0 + kTile > p.S) {
                const int lim_c = p.S - kv0;
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c >= lim_c) s[c] = -INFINITY;  // key past the end
            }
            if constexpr (E) {
                // Key kv0 + c is kept when bit c % 8 of byte c / 8 of the row's
                // 16 bytes for this key tile is set (nothing to do when all are).
                if ((keep.x & keep.y & keep.z & keep.w) != 0xFFFFFFFFu) {
                    const uint32_t kw[4] = {keep.x, keep.y, keep.z, keep.w};
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (((kw[c >> 5] >> (c & 31)) & 1u) == 0u) s[c] = -INFINITY;
                }
            }
            float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
            for (int c = 0; c < 128; c += 8) {
                mx0 = ptx::max3(mx0, s[c], s[c + 1]);
                mx1 = ptx::max3(mx1, s[c + 2], s[c + 3]);
                mx2 = ptx::max3(mx2, s[c + 4], s[c + 5]);
                mx3 = ptx::max3(mx3, s[c + 6], s[c + 7]);
            }
            const float mt = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
            // Without an element mask every row has at least one unmasked key in
            // every tile it visits (all keys of an off-diagonal tile; the first
            // key of a diagonal tile; key kv0 < S of the last tile), so mt is
            // finite.  With one, mt = -inf when the tile shows the row nothing:
            // the reference maximum stays unset (its finite initial value makes
            // every probability 0) until a tile shows a key.
            float alpha = 1.f;
            bool rescale = false;
            if (first) {
                if (!E || mt > -INFINITY) {
                    m_run = mt;
                    first = false;
                }
            } else if (mt > m_run + kRescaleSlack) {
                alpha = ptx::ex2(m_run - mt);
                m_run = mt;
                rescale = true;
            }
            // p = 2^(s*scale*log2e - m), two elements per paired FMA / add.
            const uint64_t sl2x2 = ptx::f2(sl2, sl2);
            const uint64_t negm2 = ptx::f2(-m_run, -m_run);
            uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
            if constexpr (F) {
                // FP8: four E4M3 probabilities per column, 64 keys per store,
                // over score columns [96,128) of S_i (already read).
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t pk[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const int e = 64 * h + 4 * c;
                        float x0, x1, x2, x3;
                        ptx::f2_split(ptx::fma2(ptx::f2(s[e], s[e + 1]), sl2x2, negm2), x0, x1);
                        ptx::f2_split(ptx::fma2(ptx::f2(s[e + 2], s[e + 3]), sl2x2, negm2), x2, x3);
                        const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
                        const float p2 = ptx::ex2(x2), p3 = ptx::ex2(x3);
                        acc[c & 3] = ptx::add2(acc[c & 3], ptx::add2(ptx::f2(p0, p1), ptx::f2(p2, p3)));
                        pk[c] = ptx::pack_e4m3x4(p0, p1, p2, p3);
                    }
                    ptx::tmem_st16(tP + 32u + 16u * h, pk);
                }
            } else if constexpr (DR) {
                // Dropout: the row sum takes every probability; the tensor core
                // gets the kept ones (the 256 / (256 - p8) factor is in o_scale).
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t pk[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const int e = 64 * h + 2 * c;
                        float x0, x1;
                        ptx::f2_split(ptx::fma2(ptx::f2(s[e], s[e + 1]), sl2x2, negm2), x0, x1);
                        const float p0 = ptx::ex2(x0);
                        const float p1 = ptx::ex2(x1);
                        acc[c & 3] = ptx::add2(acc[c & 3], ptx::f2(p0, p1));
                        // keys e, e+1: bytes 2 (c mod 2), 2 (c mod 2) + 1 of word e / 4
                        const uint32_t keep = pair_mask(gw[e >> 2], (c & 1) ? 0xBBAAu : 0x9988u);
                        pk[c] = ptx::pack_bf16x2(p0, p1) & keep;
                    }
                    ptx::tmem_st32(tP + 32 * h, pk);
                }
            } else {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t pk[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const int e = 64 * h + 2 * c;
                        float x0, x1;
                        ptx::f2_split(ptx::fma2(ptx::f2(s[e], s[e + 1]), sl2x2, negm2), x0, x1);
                        const float p0 = ptx::ex2(x0);
                        const float p1 = ptx::ex2(x1);
                        acc[c & 3] = ptx::add2(acc[c & 3], ptx::f2(p0, p1));
                        pk[c] = ptx::pack_bf16x2(p0, p1);
                    }
                    ptx::tmem_st32(tP + 32 * h, pk);
                }
            }
            float sum0, sum1, sum2, sum3, sum4, sum5, sum6, sum7;
            ptx::f2_split(acc[0], sum0, sum1);
            ptx::f2_split(acc[1], sum2, sum3);
            ptx::f2_split(acc[2], sum4, sum5);
            ptx::f2_split(acc[3], sum6, sum7);
            sum0 = (sum0 + sum1) + (sum2 + sum3);
            sum1 = (sum4 + sum5) + (sum6 + sum7);
            l_run = l_run * alpha + (sum0 + sum1);
            if (__any_sync(0xffffffffu, rescale)) {
                // O_i holds the sum over earlier tiles; its last MMA completed
                // before S_i(j) did.
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    ptx::tmem_ld32(tO + c * 32, o);
                    ptx::tmem_ld_wait();
                    ptx::reg_fence32(o);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    ptx::tmem_st32(tO + c * 32, o);
                }
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(bar_p);  // one arrival per warp
        }

        // ---- epilogue: wait for the last O_i += P V, then O / l -> bf16, LSE
        bool ok = ptx::mbar_wait(bar_o, o_phase, abort_flag, p.status, lim);
        if (!__all_sync(0xffffffffu, ok)) return;
        o_phase ^= 1u;
        ptx::tc_fence_after();
        const int row = qt * kTile + r;
        const bool valid = row < p.S;
        __nv_bfloat16* orow = p.out + ((size_t)w.bh * p.S + row) * D;
        // A row that sees no key (a block mask keeping no key tile of the query
        // tile, or an element mask) gets O = 0 and LSE = -inf.  When no row of
        // the warp sees a key, TMEM O is not read (with a block mask it was
        // never written); otherwise the tensor-memory loads stay warp-wide and
        // such rows write zeros.
        const bool none = (M || E) && __all_sync(0xffffffffu, first);
        if (none) {
            if (valid) {
#pragma unroll 1
                for (int c = 0; c < D; c += 8)
                    *reinterpret_cast<uint4*>(orow + c) = make_uint4(0u, 0u, 0u, 0u);
                if (p.lse != nullptr) p.lse[(size_t)w.bh * p.S + row] = -INFINITY;
            }
            if constexpr (M) {
                __syncwarp();
                if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(ws_bar<D, F>(base, L::kOEmpty + wg));
            }
            continue;
        }
        const bool row_none = E && first;  // (only element masks leave single rows empty)
        const float inv_l = row_none ? 0.f : p.o_scale / l_run;  // o_scale: the V descale (1 for bf16)
        // O / l -> bf16 -> this warp's staging box (rows 32 w .. 32 w + 31 of the
        // tile, 64 columns at a time, swizzled as the tensor map expects) -> one
        // TMA store per block; rows past S are clipped by the tensor map.
        const int row0 = qt * kTile + 32 * warp_in_wg;
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {
            // The store issued from the box before (previous block or unit) has read it.
            if (lane == 0) ptx::bulk_wait_group_read<0>();
            __syncwarp();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t o[32];
                ptx::tmem_ld32(tO + 64 * c + 32 * h, o);
                ptx::tmem_ld_wait();
                ptx::reg_fence32(o);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    uint32_t v[4];
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        v[t] = ptx::pack_bf16x2(__uint_as_float(o[8 * e + 2 * t]) * inv_l,
                                                __uint_as_float(o[8 * e + 2 * t + 1]) * inv_l);
                    // 16-byte piece 4h+e of this row, at its swizzled position.
                    ptx::st_shared_v4(stage + (uint32_t)lane * 128u + ((uint32_t)((4 * h + e) ^ (lane & 7)) << 4),
                                      v[0], v[1], v[2], v[3]);
                }
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (row0 < p.S) ptx::tma_store_3d_hint(tm_o, stage, 64 * c, row0, w.bh, written_once);
                ptx::bulk_commit_group();
            }
        }
        if (valid && p.lse != nullptr)
            p.lse[(size_t)w.bh * p.S + row] = row_none ? -INFINITY : (m_run + ptx::lg2(l_run)) * kLn2;
        if constexpr (M) {  // O_i read out: the next unit may produce its own
            ptx::tc_fence_before();
            __syncwarp();
            if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(ws_bar<D, F>(base, L::kOEmpty + wg));
        }
    }
}

// The softmax role plus the completion of this warp's output stores, which
// must have finished reading shared memory before the CTA exits.
template <int D, bool F, bool M, bool DR, bool E>
__device__ void ws_softmax_warp(const CUtensorMap* tm_o, const FwdParams& p, const FwdSchedule& sc, uint32_t base,
                                uint32_t tmem, int wg, volatile int* abort_flag) {
    ws_softmax_role<D, F, M, DR, E>(tm_o, p, sc, base, tmem, wg, abort_flag);
    if ((threadIdx.x & 31) == 0) ptx::bulk_wait_group<0>();
    __syncwarp();
}

// ---------------------------------------------------------------- kernel
template <int D, bool F, bool M, bool DR, bool E>
__global__ void __launch_bounds__(WsLayout<D, F>::kThreads, 1)
    attn_fwd_ws_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_o, const FwdParams p,
                       const __grid_constant__ FwdSchedule sched) {
    using L = WsLayout<D, F>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(ws_bar<D, F>(base, L::kQFull + i), 1);
            ptx::mbar_init(ws_bar<D, F>(base, L::kQEmpty + i), 1);
            ptx::mbar_init(ws_bar<D, F>(base, L::kSFull + i), 1);
            ptx::mbar_init(ws_bar<D, F>(base, L::kPFull + i), 4);  // one per softmax warp
            ptx::mbar_init(ws_bar<D, F>(base, L::kOFull + i), 1);
        }
        for (int s = 0; s < L::kStages; ++s) {
            ptx::mbar_init(ws_bar<D, F>(base, L::kKVFull + s), 1);
            ptx::mbar_init(ws_bar<D, F>(base, L::kKVEmpty + s), 1);
        }
        ptx::mbar_init(ws_bar<D, F>(base, L::kDrain), 1);
        for (int i = 0; i < 2; ++i) ptx::mbar_init(ws_bar<D, F>(base, L::kOEmpty + i), 4);  // one per softmax warp
        *abort_flag = 0;
        ptx::fence_barrier_init();
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        ptx::prefetch_tensormap(&tm_o);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), L::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
        ptx::regs_dec<L::kRegsSmall>();
        if (warp == 0) {
            if (lane == 0) ws_load_role<D, F, M, DR, E>(&tm_q, &tm_k, &tm_v, p, sched, base, abort_flag);
        } else if (warp == 1) {
            if (lane == 0) ws_mma_role<D, F, M, DR, E>(p, sched, base, tmem, abort_flag);
        }
    } else {
        ptx::regs_inc<L::kRegsSoftmax>();
        ws_softmax_warp<D, F, M, DR, E>(&tm_o, p, sched, base, tmem, (warp - 4) >> 2, abort_flag);
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, L::kTmemCols);
    }
}

}  // namespace attn
