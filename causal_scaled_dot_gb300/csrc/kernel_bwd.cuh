// kernel_bwd.cuh -- attention backward (dQ, dK, dV) for sm_103a.
//
// The gradients of O = softmax(scale * Q K^T, causal) V for an upstream dO:
//   P_ij    = exp(scale * q_i . k_j - LSE_i)         (the forward's weights)
//   dP_ij   = dO_i . V_j
//   delta_i = sum_j P_ij dP_ij = dO_i . O_i
//   dS_ij   = P_ij (dP_ij - delta_i)
//   dQ_i = scale * sum_j dS_ij K_j,  dK_j = scale * sum_i dS_ij Q_i,  dV_j = sum_i P_ij dO_i
// (the ai-manual.ru article, section 6, names the backward pass as the part of
// fused attention that is hard to get right; the formulas are the derivative
// of the forward, restated here, with P recomputed from the saved LSE as the
// "Profiling in PyTorch (Part 3)" retelling describes for FlashAttention,
// section "The Flash Backend": nothing of size S x S is stored).
//
// Two persistent kernels, no atomics and no scratch:
//
//  attn_bwd_dq_kernel   unit = (b, hq, query tile i), key tiles j <= i.
//     Tensor memory: S [0,128), dP [128,256), dQ [256,256+D).  Per key tile:
//     S = Q K_j^T and dP = dO V_j^T (both operands in shared memory), then
//     dQ += dS K_j with dS (bf16) read from tensor memory.  It also computes
//     delta_i = dO_i . O_i for its rows and writes it out for the second kernel.
//
//  attn_bwd_dkdv_kernel unit = (b, hkv, key tile j), over the query tiles
//     i >= j of every query head of the group (Q_i and dO_i stream through a
//     ring of single-tile slots).  Tensor memory: S^T [0,128),
//     dP^T [128,256), dV [256,256+D), dK [256+D,256+2D) -- all 512 columns at
//     D = 128.  Per query tile: S^T = K Q_i^T and dP^T = V dO_i^T, then
//     dV += P^T dO_i and dK += dS^T Q_i with P^T and dS^T read from tensor
//     memory.
//
// Roles (384 threads, 12 warps), as in the forward kernel: warp 0 TMA
// producer, warp 1 MMA issuer (one thread) and TMEM owner, warps 4-7 and 8-11
// two element-wise warpgroups.  Both warpgroups work on the same tile, one
// thread per tensor-memory lane (a row of S, or of S^T), warpgroup w on
// columns [64w, 64w+64).  Each writes its bf16 P or dS over the first half of
// its own fp32 columns, so the tensor core reads 64 columns of packed pairs
// per warpgroup.  Warps 2-3 stage per-query rows in shared memory ahead of
// use: in the dQ kernel LSE and delta_i = dO_i . O_i (computed there from
// global O and dO), in the dK/dV kernel LSE and delta of each query tile.
//
// Template flags: M, a block mask (dropped tiles are neither loaded nor
// computed; units without kept tiles write zeros); E, per-pair keep bits (the
// dQ element-wise threads read their row's bytes a key tile ahead, the dK/dV
// statistics warps stage each query tile's bytes in shared memory); DR,
// dropout of the weights with the forward's Philox keep decisions regenerated
// (in the dQ kernel per row, in the dK/dV kernel by all 256 element-wise
// threads into shared memory), dV taking the kept weights times
// 256 / (256 - p8) and dP of a dropped weight being 0.
//
// Every wait is bounded (ptx::mbar_wait); after a timeout each role returns,
// the producer first letting its issued copies land, the MMA issuer its
// issued products complete, so that the CTA can release its memory.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "philox.cuh"
#include "ptx.cuh"

namespace attn {

struct BwdParams {
    int B, Hq, Hkv, S;
    int group;       // Hq / Hkv
    int num_tiles;   // ceil(S / kTile)
    int causal;
    float scale;       // dQ, dK factor
    float scale_log2;  // scale * log2(e)
    const __nv_bfloat16* out;   // O  [B,Hq,S,D] (dQ kernel: delta)
    const __nv_bfloat16* dout;  // dO [B,Hq,S,D] (dQ kernel: delta)
    const float* lse;           // [B,Hq,S], natural log
    float* delta;               // [B,Hq,S]: written by the dQ kernel, read by the dK/dV kernel
    __nv_bfloat16* dq;          // [B,Hq,S,D]
    __nv_bfloat16* dk;          // [B,Hkv,S,D]
    __nv_bfloat16* dv;          // [B,Hkv,S,D]
    unsigned int* status;
    unsigned long long wait_limit_ns;
    int num_units;
    int head_block;  // heads worked on together (see split_unit)
    const uint8_t* block_mask;  // masked kernels: [mask_heads][nt][nt], 0 drops a (query, key) tile
    int mask_heads;             // 1 or Hq
    const uint8_t* keep_bits;   // element-masked kernels: [keep_heads][S][keep_row_bytes]
    int keep_heads;             // 1 or Hq
    int keep_row_bytes;         // 16 per 128 keys
    // Dropout kernels: weight (i, j) of head bh kept when byte j % 16 of the
    // Philox4x32-10 block {j / 16, i, bh, offset} under key {seed_lo, seed_hi}
    // is >= p8 (philox.cuh); kept weights are scaled by ks = 256 / (256 - p8)
    // (as in the forward).  The kernels fold ks into the weights,
    // P ks = 2^(s * scale_log2 - (LSE log2 e - log2 ks)), and with them
    // dS = P (Z ks dP - delta) = (P ks) (Z dP - delta / ks).
    int dropout_p8;
    unsigned long long dropout_seed, dropout_offset;
    unsigned int philox_round_keys[20];  // the key schedule of dropout_seed (philox_round_keys)
    float log2_keep_scale;  // log2(ks)
    float inv_keep_scale;   // (256 - p8) / 256, exact
};

// Block mask entry of (query head bh, query tile qt, key tile kt).
__device__ __forceinline__ bool bwd_tile_kept(const BwdParams& p, int bh, int qt, int kt) {
    const int nt = p.num_tiles;
    const int h = p.mask_heads == 1 ? 0 : bh % p.Hq;
    return __ldg(p.block_mask + ((size_t)h * nt + qt) * nt + kt) != 0;
}

// Units are (head, tile) pairs.  Heads are taken `head_block` at a time, about
// one tile of each head per CTA, so the CTAs running together share the
// streamed operands of a few heads in L2; within a block the tile index `rank`
// runs from the heaviest tile down, the head index fastest.
__device__ __forceinline__ void split_unit(int u, int heads, int tiles, int head_block, int& head,
                                           int& rank) {
    const int per_block = head_block * tiles;
    const int blk = u / per_block;
    const int within = u - blk * per_block;
    const int first = blk * head_block;
    const int hb = min(head_block, heads - first);
    rank = within / hb;
    head = first + (within - rank * hb);
}

// The unit this CTA runs in round r: boustrophedon over the CTAs, so sorted
// unit costs (heaviest first) spread evenly.
__device__ __forceinline__ int bwd_unit_of_round(int r) {
    const int G = gridDim.x, c = blockIdx.x;
    return r * G + ((r & 1) ? (G - 1 - c) : c);
}

// The dQ kernel's producer walks a second position kPrefetch key tiles ahead
// of its loads (across unit boundaries) and prefetches the tiles there into
// L2, so that the loads themselves mostly hit L2.  (The same in the dK/dV
// kernel measured slower.)
constexpr int kPrefetch = 3;
struct StreamPos {
    int rnd, u, i;  // round, unit, step within the unit
};

// ====================================================================== dQ
template <int D>
struct DqLayout {
    static constexpr int kThreads = 384;
    static constexpr int kRegsSmall = 64;
    static constexpr int kRegsWork = 216;
    static_assert(128 * kRegsSmall + 256 * kRegsWork <= kThreads * 168, "register split");
    static constexpr uint32_t kTileBytes = kTile * D * 2;
    static constexpr int kChunks = D / 64;
    static constexpr uint32_t kChunkBytes = kTile * 128;
    // K/V ring, one tile per slot.  A fifth slot at D = 128 measured slower
    // (it leaves L1 too small for the row loads).
    static constexpr int kStages = (kTileBytes == 32768) ? 4 : 8;
    static constexpr int kStatStages = 2;                  // per-row LSE / delta of a unit
    static constexpr uint32_t kStatBytes = 2 * kTile * 4;  // stage s: lse2[128], delta[128]
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kDO = kTileBytes;
    static constexpr uint32_t kRing = 2 * kTileBytes;
    static constexpr uint32_t kStat = kRing + kStages * kTileBytes;
    static constexpr uint32_t kBars = kStat + kStatStages * kStatBytes;
    static constexpr int kQFull = 0, kQEmpty = 1, kSFull = 2, kDPFull = 3, kSFree = 4, kDSFull = 5,
                         kDQFull = 6, kKVFull = 7, kKVEmpty = 7 + kStages, kStatFull = 7 + 2 * kStages,
                         kStatEmpty = 7 + 2 * kStages + kStatStages,
                         kDrain = 7 + 2 * kStages + 2 * kStatStages,
                         kDQEmpty = kDrain + 1;  // block-masked kernels: dQ read out
    static constexpr int kNumBars = kDrain + 2;
    static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kDynamicSmem = kAbort + 4 + 1024;
    static_assert(kDynamicSmem <= 227 * 1024, "shared memory budget");
};

struct DqUnit {
    int bh, kv_bh, qt, n;
};
__device__ __forceinline__ DqUnit dq_decode(int u, const BwdParams& p) {
    DqUnit w;
    int rank;
    split_unit(u, p.B * p.Hq, p.num_tiles, p.head_block, w.bh, rank);
    w.qt = p.num_tiles - 1 - rank;  // heaviest (last) query tiles first
    const int b = w.bh / p.Hq, hq = w.bh - b * p.Hq;
    w.kv_bh = b * p.Hkv + hq / p.group;
    w.n = p.causal ? w.qt + 1 : p.num_tiles;
    return w;
}

// The key tile after j that query tile w.qt uses (w.n if none): every tile
// below the causal bound, or with a block mask (M) the kept ones.
template <bool M>
__device__ __forceinline__ int dq_next_key(const BwdParams& p, const DqUnit& w, int j) {
    for (++j; j < w.n; ++j)
        if (!M || bwd_tile_kept(p, w.bh, w.qt, j)) return j;
    return w.n;
}

template <int D>
__device__ __forceinline__ uint32_t dq_bar(uint32_t base, int i) {
    return base + DqLayout<D>::kBars + 8u * (uint32_t)i;
}

template <int D, bool M, bool E, bool DR>
__device__ void dq_load_role(const CUtensorMap* tm_q, const CUtensorMap* tm_do,
                             const CUtensorMap* tm_k, const CUtensorMap* tm_v, const BwdParams& p,
                             uint32_t base, volatile int* abort_flag) {
    using L = DqLayout<D>;
    const uint64_t lim = p.wait_limit_ns;
    uint32_t qe_phase = 0, ring_phase = 0;
    int slot = 0;
    // Copies issued and possibly not landed yet, for the drain after an abort.
    bool pend_q = false;
    uint32_t pend_q_par = 0, pend_kv = 0, pend_kv_par = 0;
    StreamPos ahead{0, bwd_unit_of_round(0), 0};
    auto advance = [&](StreamPos& a) {
        if (a.u >= p.num_units) return;
        if (++a.i >= dq_decode(a.u, p).n) {
            a.i = 0;
            a.u = bwd_unit_of_round(++a.rnd);
        }
    };
    auto prefetch = [&](const StreamPos& a) {  // K_i, V_i (and Q, dO at a unit's start)
        if (a.u >= p.num_units) return;
        const DqUnit x = dq_decode(a.u, p);
        if (a.i == 0) {
            for (int c = 0; c < L::kChunks; ++c) {
                ptx::tma_prefetch_l2_3d(tm_q, c * 64, x.qt * kTile, x.bh);
                ptx::tma_prefetch_l2_3d(tm_do, c * 64, x.qt * kTile, x.bh);
            }
        }
        for (int c = 0; c < L::kChunks; ++c) {
            ptx::tma_prefetch_l2_3d(tm_k, c * 64, a.i * kTile, x.kv_bh);
            ptx::tma_prefetch_l2_3d(tm_v, c * 64, a.i * kTile, x.kv_bh);
        }
    };
    for (int k = 0; k < kPrefetch; ++k) advance(ahead);
    for (int rnd = 0, u = bwd_unit_of_round(0); u < p.num_units; u = bwd_unit_of_round(++rnd)) {
        const DqUnit w = dq_decode(u, p);
        if (!ptx::mbar_wait(dq_bar<D>(base, L::kQEmpty), qe_phase ^ 1u, abort_flag, p.status, lim))
            goto drain;
        {
            const uint32_t full = dq_bar<D>(base, L::kQFull);
            ptx::mbar_arrive_expect_tx(full, 2 * L::kTileBytes);
#pragma unroll
            for (int c = 0; c < L::kChunks; ++c) {
                ptx::tma_load_3d(base + L::kQ + c * L::kChunkBytes, tm_q, full, c * 64, w.qt * kTile, w.bh);
                ptx::tma_load_3d(base + L::kDO + c * L::kChunkBytes, tm_do, full, c * 64, w.qt * kTile, w.bh);
            }
            pend_q = true;
            pend_q_par = qe_phase;
            qe_phase ^= 1u;
        }
        for (int j = dq_next_key<M>(p, w, -1); j < w.n; j = dq_next_key<M>(p, w, j)) {
            if constexpr (!M) {
                prefetch(ahead);
                advance(ahead);
            }
#pragma unroll
            for (int t = 0; t < 2; ++t) {  // K_j, then V_j
                if (!ptx::mbar_wait(dq_bar<D>(base, L::kKVEmpty + slot), ring_phase ^ 1u, abort_flag,
                                    p.status, lim))
                    goto drain;
                const uint32_t full = dq_bar<D>(base, L::kKVFull + slot);
                ptx::mbar_arrive_expect_tx(full, L::kTileBytes);
                const CUtensorMap* map = t == 0 ? tm_k : tm_v;
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c)
                    ptx::tma_load_3d(base + L::kRing + (uint32_t)slot * L::kTileBytes + c * L::kChunkBytes,
                                     map, full, c * 64, j * kTile, w.kv_bh);
                pend_kv |= 1u << slot;
                pend_kv_par = (pend_kv_par & ~(1u << slot)) | (ring_phase << slot);
                if (++slot == L::kStages) {
                    slot = 0;
                    ring_phase ^= 1u;
                }
            }
        }
    }
    return;
drain:
    for (int s = 0; s < L::kStages; ++s)
        if (pend_kv & (1u << s))
            ptx::drain_wait(dq_bar<D>(base, L::kKVFull + s), (pend_kv_par >> s) & 1u, lim);
    if (pend_q) ptx::drain_wait(dq_bar<D>(base, L::kQFull), pend_q_par, lim);
}

// The MMA issuers of both kernels spin on their barriers (mbar_wait_spin) as
// the forward's does: the tensor core idles while its only feeding thread waits.
template <int D, bool M, bool E, bool DR>
__device__ void dq_mma_role(const BwdParams& p, uint32_t base, uint32_t tmem, volatile int* abort_flag) {
    using L = DqLayout<D>;
    constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(kTile, kTile, false);  // S, dP: N = 128 keys
    constexpr uint32_t kIdescQ = ptx::idesc_bf16_f32(kTile, D, true);       // dQ: N = D, K MN-major
    const uint64_t lim = p.wait_limit_ns;
    uint32_t qf_phase = 0, sfree_phase = 0, ds_phase = 0, ring_phase = 0;
    // Block-masked kernels: a unit without key tiles makes no handshake with the
    // element-wise warps, so before dQ of a unit is produced (or declared zero)
    // the previous unit's dQ must have been read out -- otherwise the DQFull
    // barrier could run two phases ahead of its waiters.
    uint32_t dqe_phase = 1u;
    int slot = 0;

    auto wait_ring = [&](int& got) -> bool {
        if (!ptx::mbar_wait_spin(dq_bar<D>(base, L::kKVFull + slot), ring_phase, abort_flag, p.status, lim))
            return false;
        got = slot;
        if (++slot == L::kStages) {
            slot = 0;
            ring_phase ^= 1u;
        }
        ptx::tc_fence_after();
        return true;
    };
    auto wait_bar = [&](int bar, uint32_t& phase) -> bool {
        if (!ptx::mbar_wait_spin(dq_bar<D>(base, bar), phase, abort_flag, p.status, lim)) return false;
        phase ^= 1u;
        ptx::tc_fence_after();
        return true;
    };
    auto slot_addr = [&](int s) { return base + L::kRing + (uint32_t)s * L::kTileBytes; };
    // D (=) A B^T over K = D with both operands K-major in shared memory.
    auto product = [&](uint32_t d, uint32_t a_smem, uint32_t b_smem) {
        const uint64_t a = ptx::sdesc_sw128(a_smem, 16, 1024);
        const uint64_t b = ptx::sdesc_sw128(b_smem, 16, 1024);
        if constexpr (D == 128)
            ptx::mma_ss_k128(d, a, b, kIdescS, 0u);
        else
            ptx::mma_ss_k64(d, a, b, kIdescS, 0u);
    };

    bool ok = true;
    for (int rnd = 0, u = bwd_unit_of_round(0); u < p.num_units && ok; u = bwd_unit_of_round(++rnd)) {
        const DqUnit w = dq_decode(u, p);
        if (!wait_bar(L::kQFull, qf_phase)) break;
        const int j0 = dq_next_key<M>(p, w, -1);
        if (M && j0 >= w.n) {  // no key tile kept: dQ is 0 (written by the element-wise warps)
            if (!wait_bar(L::kDQEmpty, dqe_phase)) break;
            ptx::mma_commit(dq_bar<D>(base, L::kQEmpty));
            ptx::mma_commit(dq_bar<D>(base, L::kDQFull));
            continue;
        }
        int ks, vs;
        if (!wait_ring(ks)) break;
        product(tmem, base + L::kQ, slot_addr(ks));  // S = Q K_j0^T
        ptx::mma_commit(dq_bar<D>(base, L::kSFull));
        if (!wait_ring(vs)) break;
        product(tmem + 128u, base + L::kDO, slot_addr(vs));  // dP = dO V_j0^T
        ptx::mma_commit(dq_bar<D>(base, L::kDPFull));
        ptx::mma_commit(dq_bar<D>(base, L::kKVEmpty + vs));
        // Q and dO are read only by S and dP: free them for the next unit as
        // soon as the last of those has been issued.
        if (dq_next_key<M>(p, w, j0) >= w.n) ptx::mma_commit(dq_bar<D>(base, L::kQEmpty));
        bool first = true;
        for (int j = j0, jn; j < w.n; j = jn, first = false) {
            jn = dq_next_key<M>(p, w, j);
            // S_j has been read: the next S may overwrite it.
            if (!(ok = wait_bar(L::kSFree, sfree_phase))) break;
            int ks_next = -1;
            if (jn < w.n) {
                if (!(ok = wait_ring(ks_next))) break;
                product(tmem, base + L::kQ, slot_addr(ks_next));
                ptx::mma_commit(dq_bar<D>(base, L::kSFull));
            }
            // dQ += dS_j K_j: dS of keys 0-63 in columns [128,160), keys 64-127 in
            // [192,224); K_j as an MN-major operand, keys 64-127 8 KB further in.
            if (!(ok = wait_bar(L::kDSFull, ds_phase))) break;
            if (M && first && !(ok = wait_bar(L::kDQEmpty, dqe_phase))) break;
            const uint64_t kd = ptx::sdesc_sw128(slot_addr(ks), L::kChunkBytes, 1024);
            ptx::mma_ts_k64(tmem + 256u, tmem + 128u, kd, kIdescQ, first ? 0u : 1u);
            ptx::mma_ts_k64(tmem + 256u, tmem + 192u, kd + 512u, kIdescQ, 1u);
            ptx::mma_commit(dq_bar<D>(base, L::kKVEmpty + ks));
            if (jn < w.n) {
                if (!(ok = wait_ring(vs))) break;
                product(tmem + 128u, base + L::kDO, slot_addr(vs));
                ptx::mma_commit(dq_bar<D>(base, L::kDPFull));
                ptx::mma_commit(dq_bar<D>(base, L::kKVEmpty + vs));
                if (dq_next_key<M>(p, w, jn) >= w.n) ptx::mma_commit(dq_bar<D>(base, L::kQEmpty));
            }
            ks = ks_next;
        }
        if (!ok) break;
        ptx::mma_commit(dq_bar<D>(base, L::kDQFull));
    }
    ptx::mma_commit(dq_bar<D>(base, L::kDrain));
    ptx::drain_wait(dq_bar<D>(base, L::kDrain), 0u, lim);
}

// delta_i = dO_i . O_i for one row, from global memory (16-byte loads).
template <int D>
__device__ __forceinline__ float row_delta(const __nv_bfloat16* o, const __nv_bfloat16* dout) {
    const uint4* a = reinterpret_cast<const uint4*>(o);
    const uint4* b = reinterpret_cast<const uint4*>(dout);
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
        const uint4 x = __ldg(a + c), y = __ldg(b + c);
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 xf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[e]));
            const float2 yf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ys[e]));
            acc0 = fmaf(xf.x, yf.x, acc0);
            acc1 = fmaf(xf.y, yf.y, acc1);
        }
    }
    return acc0 + acc1;
}

// Warps 2-3: for each unit, the LSE (as log2) and delta_i = dO_i . O_i of its
// 128 rows into a shared-memory stage (delta also to global memory for the
// dK/dV kernel), ahead of the element-wise warps.
template <int D, bool M, bool E, bool DR>
__device__ void dq_stat_role(const BwdParams& p, uint32_t base, uint8_t* smem, volatile int* abort_flag) {
    using L = DqLayout<D>;
    const int tid = threadIdx.x - 64;  // 0..63
    const uint64_t lim = p.wait_limit_ns;
    uint32_t ring_phase = 0;
    int st = 0;
    for (int rnd = 0, u = bwd_unit_of_round(0); u < p.num_units; u = bwd_unit_of_round(++rnd)) {
        const DqUnit w = dq_decode(u, p);
        float l2[2], dl[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = w.qt * kTile + tid + 64 * h;
            l2[h] = 0.f;
            dl[h] = 0.f;
            if (row < p.S) {
                const size_t ro = (size_t)w.bh * p.S + row;
                l2[h] = __ldg(p.lse + ro) * kLog2e;
                dl[h] = row_delta<D>(p.out + ro * D, p.dout + ro * D);
                p.delta[ro] = dl[h];
            }
        }
        if (!ptx::mbar_wait(dq_bar<D>(base, L::kStatEmpty + st), ring_phase ^ 1u, abort_flag, p.status, lim))
            return;
        float* rows = reinterpret_cast<float*>(smem + L::kStat + (uint32_t)st * L::kStatBytes);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            rows[tid + 64 * h] = l2[h];
            rows[kTile + tid + 64 * h] = dl[h];
        }
        ptx::mbar_arrive(dq_bar<D>(base, L::kStatFull + st));
        if (++st == L::kStatStages) {
            st = 0;
            ring_phase ^= 1u;
        }
    }
}

// The element-wise warps' wait for a product (S, dP): suspend-hinted, except
// in the dropout kernels, whose warps spin (same-call A/B: the backward with
// dropout 1097.5 -> 1080.7 us at B4 H16 S4096 D128, the plain one 810.8 ->
// 816.7 us with spinning, so only the dropout kernels spin).
template <bool DR>
__device__ __forceinline__ bool ew_wait_product(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                unsigned int* status, uint64_t lim) {
    if constexpr (DR)
        return ptx::mbar_wait_spin(bar, parity, abort_flag, status, lim);
    else
        return ptx::mbar_wait(bar, parity, abort_flag, status, lim);
}

template <int D, bool M, bool E, bool DR>
__device__ void dq_work_role(const BwdParams& p, uint32_t base, const uint8_t* smem, uint32_t tmem,
                             int wg, volatile int* abort_flag) {
    using L = DqLayout<D>;
    const int warp = threadIdx.x >> 5;
    const int r = (warp & 3) * 32 + (threadIdx.x & 31);  // row of the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + 64u * (uint32_t)wg;
    const uint32_t tDP = tmem + lane_off + 128u + 64u * (uint32_t)wg;  // dS (bf16) written over it
    const uint32_t tDQ = tmem + lane_off + 256u + (uint32_t)(wg * (D / 2));
    const float sl2 = p.scale_log2;
    const uint64_t lim = p.wait_limit_ns;
    uint32_t s_phase = 0, dp_phase = 0, dq_phase = 0, stat_phase = 0;
    int st = 0;

    for (int rnd = 0, u = bwd_unit_of_round(0); u < p.num_units; u = bwd_unit_of_round(++rnd)) {
        const DqUnit w = dq_decode(u, p);
        const int row = w.qt * kTile + r;
        const bool valid = row < p.S;
        const size_t ro = (size_t)w.bh * p.S + row;
        // This row's LSE (log2) and delta from the stat warps.
        {
            const bool ok = ptx::mbar_wait(dq_bar<D>(base, L::kStatFull + st), stat_phase, abort_flag,
                                           p.status, lim);
            if (!__all_sync(0xffffffffu, ok)) return;
        }
        const float* rows = reinterpret_cast<const float*>(smem + L::kStat + (uint32_t)st * L::kStatBytes);
        // Dropout: the weights come out already scaled by ks, and delta
        // is divided by it (BwdParams::log2_keep_scale).
        const float lse2 = DR ? rows[r] - p.log2_keep_scale : rows[r];
        const float delta = DR ? rows[kTile + r] * p.inv_keep_scale : rows[kTile + r];
        __syncwarp();
        if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(dq_bar<D>(base, L::kStatEmpty + st));
        if (++st == L::kStatStages) {
            st = 0;
            stat_phase ^= 1u;
        }
        const bool none = M && dq_next_key<M>(p, w, -1) >= w.n;  // no key tile kept: dQ = 0
        // Element-masked kernels: this row's 8 keep bytes for the warpgroup's 64
        // keys of each key tile, read one key tile ahead.
        const uint8_t* keep_row = nullptr;
        uint2 keep_next = make_uint2(~0u, ~0u);
        int keep_next_j = -1;
        if constexpr (E) {
            if (valid)
                keep_row = p.keep_bits +
                           ((size_t)(p.keep_heads == 1 ? 0 : w.bh % p.Hq) * p.S + row) * (size_t)p.keep_row_bytes +
                           8 * wg;
        }
        for (int j = dq_next_key<M>(p, w, -1); j < w.n; j = dq_next_key<M>(p, w, j)) {
            uint2 keep = make_uint2(~0u, ~0u);
            if constexpr (E) {
                if (keep_row != nullptr) {
                    keep = keep_next_j == j ? keep_next : __ldg(reinterpret_cast<const uint2*>(keep_row + 16 * j));
                    const int jn = dq_next_key<M>(p, w, j);
                    if (jn < w.n) {
                        keep_next = __ldg(reinterpret_cast<const uint2*>(keep_row + 16 * jn));
                        keep_next_j = jn;
                    }
                }
            }
            bool ok = ew_wait_product<DR>(dq_bar<D>(base, L::kSFull), s_phase, abort_flag, p.status, lim);
            if (!__all_sync(0xffffffffu, ok)) return;
            s_phase ^= 1u;
            ptx::tc_fence_after();
            uint32_t sr[64];
            ptx::tmem_ld32(tS, sr);
            ptx::tmem_ld32(tS + 32u, sr + 32);
            ptx::tmem_ld_wait();
            ptx::reg_fence32(sr);
            ptx::reg_fence32(sr + 32);
            // S has been read: let the tensor core overwrite it.
            ptx::tc_fence_before();
            __syncwarp();
            if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(dq_bar<D>(base, L::kSFree));

            // P = 2^(s * scale * log2 e - LSE log2 e); masked keys get 0.
            float pr[64];
            const int key0 = j * kTile + 64 * wg;
#pragma unroll
            for (int c = 0; c < 64; ++c) pr[c] = ptx::ex2(fmaf(__uint_as_float(sr[c]), sl2, -lse2));
            if (p.causal && j == w.qt) {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (64 * wg + c > r) pr[c] = 0.f;  // key after the query
            } else if (!p.causal && key0 + 64 > p.S) {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (key0 + c >= p.S) pr[c] = 0.f;  // key past the end
            }
            if constexpr (E) {  // keys whose keep bit is 0 (a row without keys has P = inf there)
                if ((keep.x & keep.y) != 0xFFFFFFFFu) {
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if ((((c < 32 ? keep.x : keep.y) >> (c & 31)) & 1u) == 0u) pr[c] = 0.f;
                }
            }
            // Dropout: keep decisions of this row's 64 keys (four Philox
            // blocks), made while the dP product runs.  A dropped weight's dP
            // is 0 (pr holds P ks, delta is delta / ks).
            uint64_t zb = ~0ull;
            if constexpr (DR) {
                zb = 0ull;
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    zb |= (uint64_t)dropout_keep16((uint32_t)((key0 >> 4) + b), (uint32_t)row, (uint32_t)w.bh,
                                                   (uint32_t)p.dropout_offset, p.philox_round_keys,
                                                   (256u - (uint32_t)p.dropout_p8) * 0x01010101u)
                          << (16 * b);
            }

            ok = ew_wait_product<DR>(dq_bar<D>(base, L::kDPFull), dp_phase, abort_flag, p.status, lim);
            if (!__all_sync(0xffffffffu, ok)) return;
            dp_phase ^= 1u;
            ptx::tc_fence_after();
            uint32_t dr[64];
            ptx::tmem_ld32(tDP, dr);
            ptx::tmem_ld32(tDP + 32u, dr + 32);
            ptx::tmem_ld_wait();
            ptx::reg_fence32(dr);
            ptx::reg_fence32(dr + 32);
            // dS = P (dP - delta), bf16 pairs over the first 32 of this
            // warpgroup's dP columns.
            auto dpd = [&](int e) {
                const float t = __uint_as_float(dr[e]) - delta;
                return (!DR || ((zb >> e) & 1ull) != 0ull) ? t : -delta;
            };
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) pk[c] = ptx::pack_bf16x2(pr[2 * c] * dpd(2 * c), pr[2 * c + 1] * dpd(2 * c + 1));
            ptx::tmem_st32(tDP, pk);
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(dq_bar<D>(base, L::kDSFull));
        }
        // Epilogue: dQ * scale -> bf16, this warpgroup's half of the columns.
        bool ok = ptx::mbar_wait(dq_bar<D>(base, L::kDQFull), dq_phase, abort_flag, p.status, lim);
        if (!__all_sync(0xffffffffu, ok)) return;
        dq_phase ^= 1u;
        ptx::tc_fence_after();
        __nv_bfloat16* drow = p.dq + ro * D + wg * (D / 2);
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {
            uint32_t o[32];
            ptx::tmem_ld32(tDQ + c * 32, o);
            ptx::tmem_ld_wait();
            ptx::reg_fence32(o);
            if (none) {
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = 0u;
            }
            if (valid) {
                uint4* dst = reinterpret_cast<uint4*>(drow + c * 32);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    uint4 v;
                    v.x = ptx::pack_bf16x2(__uint_as_float(o[8 * e + 0]) * p.scale,
                                           __uint_as_float(o[8 * e + 1]) * p.scale);
                    v.y = ptx::pack_bf16x2(__uint_as_float(o[8 * e + 2]) * p.scale,
                                           __uint_as_float(o[8 * e + 3]) * p.scale);
                    v.z = ptx::pack_bf16x2(__uint_as_float(o[8 * e + 4]) * p.scale,
                                           __uint_as_float(o[8 * e + 5]) * p.scale);
                    v.w = ptx::pack_bf16x2(__uint_as_float(o[8 * e + 6]) * p.scale,
                                           __uint_as_float(o[8 * e + 7]) * p.scale);
                    dst[e] = v;
                }
            }
        }
        if constexpr (M) {  // dQ read out: the next unit may produce its own
            ptx::tc_fence_before();
            __syncwarp();
            if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(dq_bar<D>(base, L::kDQEmpty));
        }
    }
}

template <int D, bool M, bool E, bool DR>
__global__ void __launch_bounds__(DqLayout<D>::kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const BwdParams p) {
    using L = DqLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        ptx::mbar_init(dq_bar<D>(base, L::kQFull), 1);
        ptx::mbar_init(dq_bar<D>(base, L::kQEmpty), 1);
        ptx::mbar_init(dq_bar<D>(base, L::kSFull), 1);
        ptx::mbar_init(dq_bar<D>(base, L::kDPFull), 1);
        ptx::mbar_init(dq_bar<D>(base, L::kSFree), 8);   // one per element-wise warp
        ptx::mbar_init(dq_bar<D>(base, L::kDSFull), 8);
        ptx::mbar_init(dq_bar<D>(base, L::kDQFull), 1);
        for (int s = 0; s < L::kStages; ++s) {
            ptx::mbar_init(dq_bar<D>(base, L::kKVFull + s), 1);
            ptx::mbar_init(dq_bar<D>(base, L::kKVEmpty + s), 1);
        }
        for (int s = 0; s < L::kStatStages; ++s) {
            ptx::mbar_init(dq_bar<D>(base, L::kStatFull + s), 64);  // one per stat thread
            ptx::mbar_init(dq_bar<D>(base, L::kStatEmpty + s), 8);  // one per element-wise warp
        }
        ptx::mbar_init(dq_bar<D>(base, L::kDrain), 1);
        ptx::mbar_init(dq_bar<D>(base, L::kDQEmpty), 8);  // one per element-wise warp
        *abort_flag = 0;
        ptx::fence_barrier_init();
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_do);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
        ptx::regs_dec<L::kRegsSmall>();
        if (warp == 0 && lane == 0) dq_load_role<D, M, E, DR>(&tm_q, &tm_do, &tm_k, &tm_v, p, base, abort_flag);
        if (warp == 1 && lane == 0) dq_mma_role<D, M, E, DR>(p, base, tmem, abort_flag);
        if (warp >= 2) dq_stat_role<D, M, E, DR>(p, base, smem, abort_flag);
    } else {
        ptx::regs_inc<L::kRegsWork>();
        dq_work_role<D, M, E, DR>(p, base, smem, tmem, (warp - 4) >> 2, abort_flag);
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

// ====================================================================== dK, dV
template <int D>
struct DkvLayout {
    static constexpr int kThreads = 384;
    static constexpr int kRegsSmall = 56;
    static constexpr int kRegsWork = 216;
    static_assert(128 * kRegsSmall + 256 * kRegsWork <= kThreads * 168, "register split");
    static constexpr uint32_t kTileBytes = kTile * D * 2;
    static constexpr int kChunks = D / 64;
    static constexpr uint32_t kChunkBytes = kTile * 128;
    static constexpr int kStatStages = 4;  // per-query LSE / delta rows
    // Stage s: lse2[128], delta[128] (fp32), then (element-masked kernels) the
    // 16 keep bytes of the unit's key tile for each of the 128 queries.
    static constexpr uint32_t kStatKeep = 2 * kTile * 4;
    static constexpr uint32_t kStatBytes = kStatKeep + kTile * 16;
    // Q_i, dO_i ring, one tile per slot: as many as fit (4 at D = 128, 10 or 11 at D = 64).
    static constexpr int kStages =
        (227 * 1024 - 2 * (int)kTileBytes - kStatStages * (int)kStatBytes - 2048) / (int)kTileBytes > 12
            ? 12
            : (227 * 1024 - 2 * (int)kTileBytes - kStatStages * (int)kStatBytes - 2048) / (int)kTileBytes;
    static constexpr uint32_t kK = 0;
    static constexpr uint32_t kV = kTileBytes;
    static constexpr uint32_t kRing = 2 * kTileBytes;
    static constexpr uint32_t kStat = kRing + kStages * kTileBytes;
    static constexpr uint32_t kBars = kStat + kStatStages * kStatBytes;
    static constexpr int kKVFull = 0, kKVEmpty = 1, kSFull = 2, kDPFull = 3, kPFull = 4, kDSFull = 5,
                         kAccFull = 6, kStFull = 7, kStEmpty = 7 + kStages, kStatFull = 7 + 2 * kStages,
                         kStatEmpty = 7 + 2 * kStages + kStatStages, kDrain = 7 + 2 * kStages + 2 * kStatStages,
                         kAccEmpty = kDrain + 1;  // block-masked kernels: dK, dV read out
    static constexpr int kNumBars = kDrain + 2;
    static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kDynamicSmem = kAbort + 4 + 1024;
    static_assert(kDynamicSmem <= 227 * 1024, "shared memory budget");
};

struct DkvUnit {
    int b, hkv, kv_bh, kt;  // key tile kt of key/value head kv_bh
    int q0, nq, n;          // query tiles q0 .. q0+nq-1 of each of the group's heads; n = group * nq
};
__device__ __forceinline__ DkvUnit dkv_decode(int u, const BwdParams& p) {
    DkvUnit w;
    split_unit(u, p.B * p.Hkv, p.num_tiles, p.head_block, w.kv_bh, w.kt);  // heaviest (first) key tiles first
    w.b = w.kv_bh / p.Hkv;
    w.hkv = w.kv_bh - w.b * p.Hkv;
    w.q0 = p.causal ? w.kt : 0;
    w.nq = p.num_tiles - w.q0;
    w.n = p.group * w.nq;
    return w;
}
// Iteration t of unit w -> (query head row bh, query tile).
__device__ __forceinline__ void dkv_iter(const DkvUnit& w, const BwdParams& p, int t, int& bh, int& qt) {
    const int g = t / w.nq;
    qt = w.q0 + (t - g * w.nq);
    bh = w.b * p.Hq + w.hkv * p.group + g;
}

// The iteration after t whose (query head, query tile) uses key tile w.kt
// (w.n if none): every iteration, or with a block mask (M) the kept ones.
template <bool M>
__device__ __forceinline__ int dkv_next(const BwdParams& p, const DkvUnit& w, int t) {
    for (++t; t < w.n; ++t) {
        if (!M) return t;
        int bh, qt;
        dkv_iter(w, p, t, bh, qt);
        if (bwd_tile_kept(p, bh, qt, w.kt)) return t;
    }
    return w.n;
}

template <class L>
__device__ __forceinline__ uint32_t dkv_bar(uint32_t base, int i) {
    return base + L::kBars + 8u * (uint32_t)i;
}

template <int D, bool M, bool E, bool DR>
__device__ void dkv_load_role(const CUtensorMap* tm_q, const CUtensorMap* tm_do,
                              const CUtensorMap* tm_k, const CUtensorMap* tm_v, const BwdParams& p,
                              uint32_t base, volatile int* abort_flag) {
    using L = DkvLayout<D>;
    const uint64_t lim = p.wait_limit_ns;
    uint32_t kve_phase = 0, ring_phase = 0;
    int slot = 0;
    bool pend_kv = false;
    uint32_t pend_kv_par = 0, pend_st = 0, pend_st_par = 0;
    for (int rnd = 0, u = bwd_unit_of_round(0); u < p.num_units; u = bwd_unit_of_round(++rnd)) {
        const DkvUnit w = dkv_decode(u, p);
        if (!ptx::mbar_wait(dkv_bar<L>(base, L::kKVEmpty), kve_phase ^ 1u, abort_flag, p.status, lim))
            goto drain;
        {
            const uint32_t full = dkv_bar<L>(base, L::kKVFull);
            ptx::mbar_arrive_expect_tx(full, 2 * L::kTileBytes);
#pragma unroll
            for (int c = 0; c < L::kChunks; ++c) {
                ptx::tma_load_3d(base + L::kK + c * L::kChunkBytes, tm_k, full, c * 64, w.kt * kTile, w.kv_bh);
                ptx::tma_load_3d(base + L::kV + c * L::kChunkBytes, tm_v, full, c * 64, w.kt * kTile, w.kv_bh);
            }
            pend_kv = true;
            pend_kv_par = kve_phase;
            kve_phase ^= 1u;
        }
        for (int t = dkv_next<M>(p, w, -1); t < w.n; t = dkv_next<M>(p, w, t)) {
            int bh, qt;
            dkv_iter(w, p, t, bh, qt);
#pragma unroll
            for (int x = 0; x < 2; ++x) {  // Q_i, then dO_i
                if (!ptx::mbar_wait(dkv_bar<L>(base, L::kStEmpty + slot), ring_phase ^ 1u, abort_flag,
                                    p.status, lim))
                    goto drain;
                const uint32_t full = dkv_bar<L>(base, L::kStFull + slot);
                ptx::mbar_arrive_expect_tx(full, L::kTileBytes);
                const CUtensorMap* map = x == 0 ? tm_q : tm_do;
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c)
                    ptx::tma_load_3d(base + L::kRing + (uint32_t)slot * L::kTileBytes + c * L::kChunkBytes,
                                     map, full, c * 64, qt * kTile, bh);
                pend_st |= 1u << slot;
                pend_st_par = (pend_st_par & ~(1u << slot)) | (ring_phase << slot);
                if (++slot == L::kStages) {
                    slot = 0;
                    ring_phase ^= 1u;
                }
            }
        }
    }
    return;
drain:
    for (int s = 0; s < L::kStages; ++s)
        if (pend_st & (1u << s))
            ptx::drain_wait(dkv_bar<L>(base, L::kStFull + s), (pend_st_par >> s) & 1u, lim);
    if (pend_kv) ptx::drain_wait(dkv_bar<L>(base, L::kKVFull), pend_kv_par, lim);
}

// Warps 2-3: LSE (as log2) and delta of each query tile into the stage's
// shared-memory rows; queries past the sequence end get +inf and 0 so that
// their weights vanish.
template <int D, bool M, bool E, bool DR>
__device__ void dkv_stat_role(const BwdParams& p, uint32_t base, uint8_t* smem, volatile int* abort_flag) {
    using L = DkvLayout<D>;
    const int tid = threadIdx.x - 64;  // 0..63
    const uint64_t lim = p.wait_limit_ns;
    uint32_t ring_phase = 0;
    int st = 0;
    for (int rnd = 0, u = bwd_unit_of_round(0); u < p.num_units; u = bwd_unit_of_round(++rnd)) {
        const DkvUnit w = dkv_decode(u, p);
        for (int t = dkv_next<M>(p, w, -1); t < w.n; t = dkv_next<M>(p, w, t)) {
            int bh, qt;
            dkv_iter(w, p, t, bh, qt);
            float l2[2], dl[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = qt * kTile + tid + 64 * h;
                const bool valid = row < p.S;
                l2[h] = valid ? __ldg(p.lse + (size_t)bh * p.S + row) * kLog2e : INFINITY;
                dl[h] = valid ? p.delta[(size_t)bh * p.S + row] : 0.f;
                if constexpr (DR) {  // weights scaled by ks, delta divided by it
                    l2[h] -= p.log2_keep_scale;
                    dl[h] *= p.inv_keep_scale;
                }
            }
            uint4 kb[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
            if constexpr (E) {  // each query's keep bits for this key tile
                const int hq = bh % p.Hq;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = qt * kTile + tid + 64 * h;
                    if (row < p.S)
                        kb[h] = __ldg(reinterpret_cast<const uint4*>(
                            p.keep_bits + ((size_t)(p.keep_heads == 1 ? 0 : hq) * p.S + row) * (size_t)p.keep_row_bytes +
                            16 * w.kt));
                }
            }
            if (!ptx::mbar_wait(dkv_bar<L>(base, L::kStatEmpty + st), ring_phase ^ 1u, abort_flag, p.status, lim))
                return;
            float* rows = reinterpret_cast<float*>(smem + L::kStat + (uint32_t)st * L::kStatBytes);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                rows[tid + 64 * h] = l2[h];
                rows[kTile + tid + 64 * h] = dl[h];
            }
            if constexpr (E) {
                uint4* keep = reinterpret_cast<uint4*>(smem + L::kStat + (uint32_t)st * L::kStatBytes + L::kStatKeep);
                keep[tid] = kb[0];
                keep[tid + 64] = kb[1];
            }
            ptx::mbar_arrive(dkv_bar<L>(base, L::kStatFull + st));
            if (++st == L::kStatStages) {
                st = 0;
                ring_phase ^= 1u;
            }
        }
    }
}

template <int D, bool M, bool E, bool DR>
__device__ void dkv_mma_role(const BwdParams& p, uint32_t base, uint32_t tmem, volatile int* abort_flag) {
    using L = DkvLayout<D>;
    constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(kTile, kTile, false);  // S^T, dP^T: N = 128 queries
    constexpr uint32_t kIdescA = ptx::idesc_bf16_f32(kTile, D, true);       // dV, dK: N = D, MN-major
    const uint64_t lim = p.wait_limit_ns;
    uint32_t kvf_phase = 0, p_phase = 0, ds_phase = 0, ring_phase = 0;
    // Block-masked kernels: as in the dQ kernel, dK and dV of the previous unit
    // must have been read out before this unit produces (or zeroes) its own.
    uint32_t acce_phase = 1u;
    int slot = 0;

    auto wait_bar = [&](int bar, uint32_t& phase) -> bool {
        if (!ptx::mbar_wait_spin(dkv_bar<L>(base, bar), phase, abort_flag, p.status, lim)) return false;
        phase ^= 1u;
        ptx::tc_fence_after();
        return true;
    };
    auto wait_ring = [&](int& got) -> bool {
        if (!ptx::mbar_wait_spin(dkv_bar<L>(base, L::kStFull + slot), ring_phase, abort_flag, p.status, lim))
            return false;
        got = slot;
        if (++slot == L::kStages) {
            slot = 0;
            ring_phase ^= 1u;
        }
        ptx::tc_fence_after();
        return true;
    };
    auto slot_addr = [&](int s) { return base + L::kRing + (uint32_t)s * L::kTileBytes; };
    auto product = [&](uint32_t d, uint32_t a_smem, uint32_t b_smem) {
        const uint64_t a = ptx::sdesc_sw128(a_smem, 16, 1024);
        const uint64_t b = ptx::sdesc_sw128(b_smem, 16, 1024);
        if constexpr (D == 128)
            ptx::mma_ss_k128(d, a, b, kIdescS, 0u);
        else
            ptx::mma_ss_k64(d, a, b, kIdescS, 0u);
    };
    const uint32_t tDV = tmem + 256u, tDK = tmem + 256u + D;

    bool ok = true;
    for (int rnd = 0, u = bwd_unit_of_round(0); u < p.num_units && ok; u = bwd_unit_of_round(++rnd)) {
        const DkvUnit w = dkv_decode(u, p);
        if (!wait_bar(L::kKVFull, kvf_phase)) break;
        const int t0 = dkv_next<M>(p, w, -1);
        if (M && t0 >= w.n) {  // no query tile keeps this key tile: dK = dV = 0
            if (!wait_bar(L::kAccEmpty, acce_phase)) break;
            ptx::mma_commit(dkv_bar<L>(base, L::kKVEmpty));
            ptx::mma_commit(dkv_bar<L>(base, L::kAccFull));
            continue;
        }
        int qs, ds, qs_next = -1, ds_next = -1;
        if (!wait_ring(qs)) break;
        product(tmem, base + L::kK, slot_addr(qs));  // S^T = K Q^T
        ptx::mma_commit(dkv_bar<L>(base, L::kSFull));
        if (!wait_ring(ds)) break;
        product(tmem + 128u, base + L::kV, slot_addr(ds));  // dP^T = V dO^T
        ptx::mma_commit(dkv_bar<L>(base, L::kDPFull));
        // K and V are read only by S^T and dP^T: free them for the next unit
        // as soon as the last of those has been issued.
        if (dkv_next<M>(p, w, t0) >= w.n) ptx::mma_commit(dkv_bar<L>(base, L::kKVEmpty));
        bool first = true;
        for (int t = t0, tn; t < w.n; t = tn, first = false) {
            tn = dkv_next<M>(p, w, t);
            // dV += P^T dO: P^T of queries 0-63 in columns [0,32), 64-127 in
            // [64,96); dO as an MN-major operand, queries 64-127 8 KB further in.
            if (!(ok = wait_bar(L::kPFull, p_phase))) break;
            if (M && first && !(ok = wait_bar(L::kAccEmpty, acce_phase))) break;
            const uint64_t dod = ptx::sdesc_sw128(slot_addr(ds), L::kChunkBytes, 1024);
            ptx::mma_ts_k64(tDV, tmem, dod, kIdescA, first ? 0u : 1u);
            ptx::mma_ts_k64(tDV, tmem + 64u, dod + 512u, kIdescA, 1u);
            ptx::mma_commit(dkv_bar<L>(base, L::kStEmpty + ds));
            if (tn < w.n) {
                if (!(ok = wait_ring(qs_next))) break;
                product(tmem, base + L::kK, slot_addr(qs_next));
                ptx::mma_commit(dkv_bar<L>(base, L::kSFull));
            }
            // dK += dS^T Q: dS^T in columns [128,160) and [192,224).
            if (!(ok = wait_bar(L::kDSFull, ds_phase))) break;
            const uint64_t qd = ptx::sdesc_sw128(slot_addr(qs), L::kChunkBytes, 1024);
            ptx::mma_ts_k64(tDK, tmem + 128u, qd, kIdescA, first ? 0u : 1u);
            ptx::mma_ts_k64(tDK, tmem + 192u, qd + 512u, kIdescA, 1u);
            ptx::mma_commit(dkv_bar<L>(base, L::kStEmpty + qs));
            if (tn < w.n) {
                if (!(ok = wait_ring(ds_next))) break;
                product(tmem + 128u, base + L::kV, slot_addr(ds_next));
                ptx::mma_commit(dkv_bar<L>(base, L::kDPFull));
                if (dkv_next<M>(p, w, tn) >= w.n) ptx::mma_commit(dkv_bar<L>(base, L::kKVEmpty));
            }
            qs = qs_next;
            ds = ds_next;
        }
        if (!ok) break;
        ptx::mma_commit(dkv_bar<L>(base, L::kAccFull));
    }
    ptx::mma_commit(dkv_bar<L>(base, L::kDrain));
    ptx::drain_wait(dkv_bar<L>(base, L::kDrain), 0u, lim);
}

template <int D, bool M, bool E, bool DR>
__device__ void dkv_work_role(const BwdParams& p, uint32_t base, const uint8_t* smem, uint32_t tmem,
                              int wg, volatile int* abort_flag) {
    using L = DkvLayout<D>;
    const int warp = threadIdx.x >> 5;
    const int r = (warp & 3) * 32 + (threadIdx.x & 31);  // key row of the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + 64u * (uint32_t)wg;          // P^T (bf16) written over it
    const uint32_t tDP = tmem + lane_off + 128u + 64u * (uint32_t)wg;  // dS^T (bf16) written over it
    const float sl2 = p.scale_log2;
    const uint64_t lim = p.wait_limit_ns;
    uint32_t s_phase = 0, dp_phase = 0, acc_phase = 0, ring_phase = 0;
    int st = 0;

    for (int rnd = 0, u = bwd_unit_of_round(0); u < p.num_units; u = bwd_unit_of_round(++rnd)) {
        const DkvUnit w = dkv_decode(u, p);
        const bool none = M && dkv_next<M>(p, w, -1) >= w.n;  // no query tile kept: dK = dV = 0
        for (int t = dkv_next<M>(p, w, -1); t < w.n; t = dkv_next<M>(p, w, t)) {
            int bh, qt;
            dkv_iter(w, p, t, bh, qt);
            // Dropout: bit c of zb keeps (query 64 wg + c, this key).  The
            // warp's 32 keys (32 (warp % 4) + k) need, for each of the
            // warpgroup's 64 queries, two 16-key Philox blocks: lane l runs the
            // four of queries 64 wg + l and 64 wg + 32 + l, as one 32-bit word
            // per query (bit k: key 32 (warp % 4) + k), and two bit transposes
            // across the warp hand every lane its own key's 64 decisions --
            // while S^T is being computed, with no exchange between warps.
            uint64_t zb = ~0ull;
            if constexpr (DR) {
                const uint32_t c4 = (256u - (uint32_t)p.dropout_p8) * 0x01010101u;
                uint32_t word[2];
#pragma unroll
                for (int y = 0; y < 2; ++y) {
                    const uint32_t query = (uint32_t)(qt * kTile + 64 * wg + 32 * y) + (threadIdx.x & 31u);
                    word[y] = 0u;
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        word[y] |= dropout_keep16((uint32_t)(w.kt * 8 + 2 * (warp & 3) + h), query, (uint32_t)bh,
                                                  (uint32_t)p.dropout_offset, p.philox_round_keys, c4)
                                   << (16 * h);
                }
                zb = (uint64_t)warp_transpose_bits(word[0]) | ((uint64_t)warp_transpose_bits(word[1]) << 32);
            }
            bool ok = ptx::mbar_wait(dkv_bar<L>(base, L::kStatFull + st), ring_phase, abort_flag, p.status, lim);
            ok = ok && ew_wait_product<DR>(dkv_bar<L>(base, L::kSFull), s_phase, abort_flag, p.status, lim);
            if (!__all_sync(0xffffffffu, ok)) return;
            s_phase ^= 1u;
            ptx::tc_fence_after();
            const float* lse2 = reinterpret_cast<const float*>(smem + L::kStat + (uint32_t)st * L::kStatBytes) + 64 * wg;
            const float* dlt = lse2 + kTile;
            uint32_t sr[64];
            ptx::tmem_ld32(tS, sr);
            ptx::tmem_ld32(tS + 32u, sr + 32);
            ptx::tmem_ld_wait();
            ptx::reg_fence32(sr);
            ptx::reg_fence32(sr + 32);
            // P^T: row = this key, columns = queries 64wg .. 64wg+63.
            float pr[64];
#pragma unroll
            for (int c = 0; c < 64; c += 4) {
                const float4 l4 = *reinterpret_cast<const float4*>(lse2 + c);
                pr[c + 0] = ptx::ex2(fmaf(__uint_as_float(sr[c + 0]), sl2, -l4.x));
                pr[c + 1] = ptx::ex2(fmaf(__uint_as_float(sr[c + 1]), sl2, -l4.y));
                pr[c + 2] = ptx::ex2(fmaf(__uint_as_float(sr[c + 2]), sl2, -l4.z));
                pr[c + 3] = ptx::ex2(fmaf(__uint_as_float(sr[c + 3]), sl2, -l4.w));
            }
            if (p.causal && qt == w.kt) {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (64 * wg + c < r) pr[c] = 0.f;  // query before this key
            }
            if constexpr (E) {
                // Query 64 wg + c keeps this key when bit r of its 16 keep bytes
                // is set: word r / 32 of that query's row in the stage, the same
                // word for the whole warp (a broadcast read).
                const uint32_t* kw = reinterpret_cast<const uint32_t*>(
                    smem + L::kStat + (uint32_t)st * L::kStatBytes + L::kStatKeep) + (r >> 5);
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (((kw[4 * (64 * wg + c)] >> (r & 31)) & 1u) == 0u) pr[c] = 0.f;
            }
            // Dropout: pr holds P ks (the stage's LSE and delta carry
            // the scaling), dV takes it where kept, and dP of a dropped weight
            // is 0.
            auto kept = [&](int c) -> bool { return !DR || ((zb >> c) & 1ull) != 0ull; };
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                if constexpr (DR)
                    pk[c] = ptx::pack_bf16x2(kept(2 * c) ? pr[2 * c] : 0.f, kept(2 * c + 1) ? pr[2 * c + 1] : 0.f);
                else
                    pk[c] = ptx::pack_bf16x2(pr[2 * c], pr[2 * c + 1]);
            }
            ptx::tmem_st32(tS, pk);
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(dkv_bar<L>(base, L::kPFull));

            ok = ew_wait_product<DR>(dkv_bar<L>(base, L::kDPFull), dp_phase, abort_flag, p.status, lim);
            if (!__all_sync(0xffffffffu, ok)) return;
            dp_phase ^= 1u;
            ptx::tc_fence_after();
            uint32_t dr[64];
            ptx::tmem_ld32(tDP, dr);
            ptx::tmem_ld32(tDP + 32u, dr + 32);
            ptx::tmem_ld_wait();
            ptx::reg_fence32(dr);
            ptx::reg_fence32(dr + 32);
#pragma unroll
            for (int c = 0; c < 64; c += 4) {
                const float4 d4 = *reinterpret_cast<const float4*>(dlt + c);
                auto dpd = [&](int e, float d) {
                    const float t = __uint_as_float(dr[e]) - d;
                    return kept(e) ? t : -d;
                };
                const float a0 = pr[c + 0] * dpd(c + 0, d4.x);
                const float a1 = pr[c + 1] * dpd(c + 1, d4.y);
                const float a2 = pr[c + 2] * dpd(c + 2, d4.z);
                const float a3 = pr[c + 3] * dpd(c + 3, d4.w);
                pk[c / 2] = ptx::pack_bf16x2(a0, a1);
                pk[c / 2 + 1] = ptx::pack_bf16x2(a2, a3);
            }
            ptx::tmem_st32(tDP, pk);
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if ((threadIdx.x & 31) == 0) {
                ptx::mbar_arrive(dkv_bar<L>(base, L::kDSFull));
                ptx::mbar_arrive(dkv_bar<L>(base, L::kStatEmpty + st));
            }
            if (++st == L::kStatStages) {
                st = 0;
                ring_phase ^= 1u;
            }
        }
        // Epilogue: warpgroup 0 writes dV, warpgroup 1 writes dK * scale.
        bool ok = ptx::mbar_wait(dkv_bar<L>(base, L::kAccFull), acc_phase, abort_flag, p.status, lim);
        if (!__all_sync(0xffffffffu, ok)) return;
        acc_phase ^= 1u;
        ptx::tc_fence_after();
        const int key = w.kt * kTile + r;
        const bool valid = key < p.S;
        const float f = wg == 0 ? 1.f : p.scale;
        __nv_bfloat16* drow = (wg == 0 ? p.dv : p.dk) + ((size_t)w.kv_bh * p.S + key) * D;
        const uint32_t tA = tmem + lane_off + 256u + (uint32_t)(wg * D);
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            ptx::tmem_ld32(tA + c * 32, o);
            ptx::tmem_ld_wait();
            ptx::reg_fence32(o);
            if (none) {
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = 0u;
            }
            if (valid) {
                uint4* dst = reinterpret_cast<uint4*>(drow + c * 32);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    uint4 v;
                    v.x = ptx::pack_bf16x2(__uint_as_float(o[8 * e + 0]) * f, __uint_as_float(o[8 * e + 1]) * f);
                    v.y = ptx::pack_bf16x2(__uint_as_float(o[8 * e + 2]) * f, __uint_as_float(o[8 * e + 3]) * f);
                    v.z = ptx::pack_bf16x2(__uint_as_float(o[8 * e + 4]) * f, __uint_as_float(o[8 * e + 5]) * f);
                    v.w = ptx::pack_bf16x2(__uint_as_float(o[8 * e + 6]) * f, __uint_as_float(o[8 * e + 7]) * f);
                    dst[e] = v;
                }
            }
        }
        if constexpr (M) {  // dK, dV read out: the next unit may produce its own
            ptx::tc_fence_before();
            __syncwarp();
            if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(dkv_bar<L>(base, L::kAccEmpty));
        }
    }
}

template <int D, bool M, bool E, bool DR>
__global__ void __launch_bounds__(DkvLayout<D>::kThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const BwdParams p) {
    using L = DkvLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        ptx::mbar_init(dkv_bar<L>(base, L::kKVFull), 1);
        ptx::mbar_init(dkv_bar<L>(base, L::kKVEmpty), 1);
        ptx::mbar_init(dkv_bar<L>(base, L::kSFull), 1);
        ptx::mbar_init(dkv_bar<L>(base, L::kDPFull), 1);
        ptx::mbar_init(dkv_bar<L>(base, L::kPFull), 8);   // one per element-wise warp
        ptx::mbar_init(dkv_bar<L>(base, L::kDSFull), 8);
        ptx::mbar_init(dkv_bar<L>(base, L::kAccFull), 1);
        for (int s = 0; s < L::kStages; ++s) {
            ptx::mbar_init(dkv_bar<L>(base, L::kStFull + s), 1);
            ptx::mbar_init(dkv_bar<L>(base, L::kStEmpty + s), 1);
        }
        for (int s = 0; s < L::kStatStages; ++s) {
            ptx::mbar_init(dkv_bar<L>(base, L::kStatFull + s), 64);  // one per loader thread
            ptx::mbar_init(dkv_bar<L>(base, L::kStatEmpty + s), 8);  // one per element-wise warp
        }
        ptx::mbar_init(dkv_bar<L>(base, L::kDrain), 1);
        ptx::mbar_init(dkv_bar<L>(base, L::kAccEmpty), 8);  // one per element-wise warp
        *abort_flag = 0;
        ptx::fence_barrier_init();
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_do);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
        ptx::regs_dec<L::kRegsSmall>();
        if (warp == 0 && lane == 0) dkv_load_role<D, M, E, DR>(&tm_q, &tm_do, &tm_k, &tm_v, p, base, abort_flag);
        if (warp == 1 && lane == 0) dkv_mma_role<D, M, E, DR>(p, base, tmem, abort_flag);
        if (warp >= 2) dkv_stat_role<D, M, E, DR>(p, base, smem, abort_flag);
    } else {
        ptx::regs_inc<L::kRegsWork>();
        dkv_work_role<D, M, E, DR>(p, base, smem, tmem, (warp - 4) >> 2, abort_flag);
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

}  // namespace attn
