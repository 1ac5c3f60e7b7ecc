// kernel_simple.cuh -- reference-structure attention forward for sm_103a.
//
// One CTA of 128 threads computes one 128-row query tile of one (batch, head)
// with no overlap between stages: TMA loads Q, K_j, V_j; one thread issues
// tcgen05.mma for S = Q K_j^T into tensor memory; every thread (one query
// row each) runs the online softmax on its TMEM lane, writes P as bf16 back
// into TMEM and rescales its O row; one thread issues O += P V_j with P read
// from TMEM.  It exists to validate the descriptor encodings and the TMEM
// layouts in the simplest possible schedule, and as a second, independently
// scheduled implementation to cross-check the pipelined kernel against.
//
// The steps are those of the naive causal attention in the "Profiling in
// PyTorch (Part 3)" retelling (section "Naive Attention": QK^T, scale,
// causal -inf mask, softmax, times V), fused with the tiled online softmax
// that the same retelling describes for FlashAttention-2 ("The Flash
// Backend"): scores never leave the SM.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace attn {

template <int D>
struct SimpleLayout {
    static constexpr uint32_t kTileBytes = kTile * D * 2;  // 32 KB at D = 128
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kK = kTileBytes;
    static constexpr uint32_t kV = 2 * kTileBytes;
    static constexpr uint32_t kBars = 3 * kTileBytes;  // 3 mbarriers
    static constexpr uint32_t kTmemSlot = kBars + 32;
    static constexpr uint32_t kAbort = kBars + 40;
    static constexpr uint32_t kBytes = kBars + 64;
    static constexpr uint32_t kDynamicSmem = kBytes + 1024;  // slack for 1024-byte alignment
    static constexpr uint32_t kTmemCols = 256;               // S/P [0,128) + O [128,128+D)
};

template <int D>
__global__ void __launch_bounds__(128, 1)
    attn_fwd_simple_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
    using L = SimpleLayout<D>;
    constexpr int kChunks = D / 64;                  // 64-column swizzle blocks across D
    constexpr uint32_t kChunkBytes = kTile * 128;    // one block of a 128-row tile: 16 KB
    constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(kTile, kTile, false);
    constexpr uint32_t kIdescO = ptx::idesc_bf16_f32(kTile, D, true);

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    const uint32_t sQ = base + L::kQ, sK = base + L::kK, sV = base + L::kV;
    const uint32_t bar_load = base + L::kBars, bar_s = bar_load + 8, bar_o = bar_load + 16;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int bh = blockIdx.x;                         // b * Hq + hq
    const int qt = p.num_q_tiles - 1 - blockIdx.y;     // heaviest causal tiles launch first
    const int b = bh / p.Hq;
    const int hq = bh - b * p.Hq;
    const int kv_bh = b * p.Hkv + hq / p.group;        // grouped-query head mapping

    if (tid == 0) {
        ptx::mbar_init(bar_load, 1);
        ptx::mbar_init(bar_s, 1);
        ptx::mbar_init(bar_o, 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), L::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_off;          // this warp's lanes, S/P columns
    const uint32_t tO = tmem + lane_off + 128;    // this warp's lanes, O columns

    const int n_kv = p.causal ? (qt + 1) : p.num_q_tiles;
    const int row = qt * kTile + tid;
    float m_run = -INFINITY;  // running max of scale*log2(e)*s over keys seen
    float l_run = 0.f;        // running sum of 2^(scale*log2(e)*s - m_run)
    uint32_t ph_load = 0, ph_s = 0, ph_o = 0;
    bool pend_load = false, pend_s = false, pend_o = false;  // thread 0: issued, not yet seen

    for (int j = 0; j < n_kv; ++j) {
        // ---- a0: TMA loads (Q once, then K_j and V_j)
        if (tid == 0 && !*abort_flag) {
            const uint32_t bytes = (j == 0 ? 3u : 2u) * L::kTileBytes;
            ptx::mbar_arrive_expect_tx(bar_load, bytes);
#pragma unroll
            for (int c = 0; c < kChunks; ++c) {
                if (j == 0) ptx::tma_load_3d(sQ + c * kChunkBytes, &tm_q, bar_load, c * 64, qt * kTile, bh);
                ptx::tma_load_3d(sK + c * kChunkBytes, &tm_k, bar_load, c * 64, j * kTile, kv_bh);
                ptx::tma_load_3d(sV + c * kChunkBytes, &tm_v, bar_load, c * 64, j * kTile, kv_bh);
            }
            pend_load = true;
        }
        if (ptx::mbar_wait(bar_load, ph_load, abort_flag, p.status, p.wait_limit_ns) && tid == 0)
            pend_load = false;
        ph_load ^= 1;

        // ---- a1: S = Q K_j^T  (M = N = 128, K = D in steps of 16)
        if (tid == 0 && !*abort_flag) {
            ptx::tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t off = (ks >> 2) * kChunkBytes + (ks & 3) * 32;
                const uint64_t a = ptx::sdesc_sw128(sQ + off, 16, 1024);
                const uint64_t bd = ptx::sdesc_sw128(sK + off, 16, 1024);
                ptx::mma_ss(tmem, a, bd, kIdescS, ks > 0 ? 1u : 0u);
            }
            ptx::mma_commit(bar_s);
            pend_s = true;
        }
        if (ptx::mbar_wait(bar_s, ph_s, abort_flag, p.status, p.wait_limit_ns) && tid == 0)
            pend_s = false;
        ph_s ^= 1;
        ptx::tc_fence_after();

        // ---- a2..a4: scale, causal mask, online softmax on this thread's row
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
                if (c > tid) s[c] = -INFINITY;  // key kv0 + c after query kv0 + tid
        } else if (!p.causal && kv0 + kTile > p.S) {
#pragma unroll
            for (int c = 0; c < 128; ++c)
                if (kv0 + c >= p.S) s[c] = -INFINITY;  // keys past the sequence end
        }
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 128; ++c) mx = fmaxf(mx, s[c]);
        const float m_new = fmaxf(m_run, mx * p.scale_log2);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ptx::ex2(m_run - m_use);
        float sum = 0.f;
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
            const float p0 = ptx::ex2(fmaf(s[2 * c], p.scale_log2, -m_use));
            const float p1 = ptx::ex2(fmaf(s[2 * c + 1], p.scale_log2, -m_use));
            sum += p0 + p1;
            pk[c] = ptx::pack_bf16x2(p0, p1);
        }
        l_run = l_run * alpha + sum;
        m_run = m_new;
        // P (bf16, 2 per column) overwrites the first 64 columns of S.
        ptx::tmem_st32(tS, pk);
        ptx::tmem_st32(tS + 32, pk + 32);
        // ---- correction: O *= alpha (O holds the previous tiles' sum)
        if (j > 0) {
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                ptx::tmem_ld32(tO + c * 32, o);
                ptx::tmem_ld_wait();
                ptx::reg_fence32(o);
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                ptx::tmem_st32(tO + c * 32, o);
            }
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncthreads();

        // ---- a5: O += P V_j  (M = 128, N = D, K = 128 keys in steps of 16)
        if (tid == 0 && !*abort_flag) {
            ptx::tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < kTile / 16; ++ks) {
                const uint64_t bd = ptx::sdesc_sw128(sV + ks * 16 * 128, kChunkBytes, 1024);
                ptx::mma_ts(tmem + 128, tmem + ks * 8, bd, kIdescO, (j > 0 || ks > 0) ? 1u : 0u);
            }
            ptx::mma_commit(bar_o);
            pend_o = true;
        }
        if (ptx::mbar_wait(bar_o, ph_o, abort_flag, p.status, p.wait_limit_ns) && tid == 0)
            pend_o = false;
        ph_o ^= 1;
        ptx::tc_fence_after();
    }

    // ---- a6: epilogue, O / l -> bf16, LSE
    const bool aborted = *abort_flag != 0;
    const float inv_l = 1.f / l_run;
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        ptx::tmem_ld32(tO + c * 32, o);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(o);
        if (row < p.S && !aborted) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
                pk[e] = ptx::pack_bf16x2(__uint_as_float(o[2 * e]) * inv_l,
                                         __uint_as_float(o[2 * e + 1]) * inv_l);
            uint4* dst = reinterpret_cast<uint4*>(p.out + ((size_t)bh * p.S + row) * D + c * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
    }
    if (row < p.S && !aborted && p.lse != nullptr)
        p.lse[(size_t)bh * p.S + row] = (m_run + ptx::lg2(l_run)) * kLn2;

    // ---- teardown: drain anything still in flight after an abort, free TMEM
    if (tid == 0 && aborted) {
        if (pend_load) ptx::drain_wait(bar_load, ph_load ^ 1, p.wait_limit_ns);
        if (pend_s) ptx::drain_wait(bar_s, ph_s ^ 1, p.wait_limit_ns);
        if (pend_o) ptx::drain_wait(bar_o, ph_o ^ 1, p.wait_limit_ns);
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, L::kTmemCols);
    }
}

}  // namespace attn
