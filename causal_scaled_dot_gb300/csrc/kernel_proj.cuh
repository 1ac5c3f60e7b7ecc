// kernel_proj.cuh -- the attention output projection on sm_103a:
//     Y[b, s, e] = sum_h sum_d O[b, h, s, d] * W[e, h*D + d] + bias[e]
// the layer's next operation after attention (the "output projection" row of
// the per-operator profile in the ainews.cool article).  O is read where the
// attention kernels leave it, [B, H, S, D]: the product's reduction index
// k = h*D + d runs over heads, so each 64-wide K chunk is one head's 128 rows
// x 64 columns, fetched by TMA straight from the [B*H, S, D] view -- no
// transpose of O to [B, S, H*D] and no intermediate buffer.
//
// Persistent tcgen05 GEMM: tiles of 128 rows (one batch entry's S positions)
// x 256 output features, K in chunks of 64 through a 4-stage TMA ring, the
// fp32 accumulator in tensor memory double-buffered (2 x 256 columns) so that
// the epilogue of one tile overlaps the products of the next.
//   warp 0      TMA producer (A chunk from O, B chunk from W)
//   warp 1      MMA issuer (M128 N256 K16, both operands in shared memory) and TMEM owner
//   warps 4-11  epilogue: warpgroup w adds the bias to columns [128w, 128w+128)
//               of a tile and stores bf16 rows of Y.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace attn {

struct ProjParams {
    int B, H, S, E;
    int m_tiles_per_batch;  // ceil(S / 128)
    int n_tiles;            // ceil(E / 256)
    int num_units;          // B * m_tiles_per_batch * n_tiles
    int k_chunks;           // H * D / 64
    const float* bias;      // [E] or null
    __nv_bfloat16* y;       // [B, S, E]
    unsigned int* status;
    unsigned long long wait_limit_ns;
};

struct ProjLayout {
    static constexpr int kThreads = 384;
    static constexpr int kRegsSmall = 56;
    static constexpr int kRegsWork = 216;
    static_assert(128 * kRegsSmall + 256 * kRegsWork <= kThreads * 168, "register split");
    static constexpr int kBM = 128, kBN = 256, kBK = 64;
    static constexpr uint32_t kABytes = kBM * kBK * 2;   // 16 KB
    static constexpr uint32_t kBBytes = kBN * kBK * 2;   // 32 KB
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr int kStages = 4;
    static constexpr uint32_t kBars = kStages * kStageBytes;
    static constexpr int kFull = 0, kEmpty = kStages, kAccFull = 2 * kStages, kAccEmpty = 2 * kStages + 2,
                         kDrain = 2 * kStages + 4;
    static constexpr int kNumBars = kDrain + 1;
    static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kDynamicSmem = kAbort + 4 + 1024;
    static_assert(kDynamicSmem <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ uint32_t proj_bar(uint32_t base, int i) {
    return base + ProjLayout::kBars + 8u * (uint32_t)i;
}

// Unit u -> (batch entry b, first row s0, first feature e0).
struct ProjUnit {
    int b, s0, e0;
};
__device__ __forceinline__ ProjUnit proj_decode(int u, const ProjParams& p) {
    const int mt = u / p.n_tiles, nt = u - (u / p.n_tiles) * p.n_tiles;
    ProjUnit w;
    w.b = mt / p.m_tiles_per_batch;
    w.s0 = (mt - w.b * p.m_tiles_per_batch) * ProjLayout::kBM;
    w.e0 = nt * ProjLayout::kBN;
    return w;
}

template <int D>
__device__ void proj_load_role(const CUtensorMap* tm_o, const CUtensorMap* tm_w, const ProjParams& p,
                               uint32_t base, volatile int* abort_flag) {
    using L = ProjLayout;
    const uint64_t lim = p.wait_limit_ns;
    int slot = 0;
    uint32_t phase = 0, pend = 0, pend_par = 0;
    for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
        const ProjUnit w = proj_decode(u, p);
        for (int kc = 0; kc < p.k_chunks; ++kc) {
            if (!ptx::mbar_wait(proj_bar(base, L::kEmpty + slot), phase ^ 1u, abort_flag, p.status, lim))
                goto drain;
            const uint32_t full = proj_bar(base, L::kFull + slot);
            ptx::mbar_arrive_expect_tx(full, L::kStageBytes);
            const uint32_t dst = base + (uint32_t)slot * L::kStageBytes;
            const int h = kc / (D / 64), d0 = (kc - h * (D / 64)) * 64;
            ptx::tma_load_3d(dst, tm_o, full, d0, w.s0, w.b * p.H + h);       // O[b, h, s0.., d0..]
            ptx::tma_load_3d(dst + L::kABytes, tm_w, full, kc * 64, w.e0, 0);  // W[e0.., kc*64..]
            pend |= 1u << slot;
            pend_par = (pend_par & ~(1u << slot)) | (phase << slot);
            if (++slot == L::kStages) {
                slot = 0;
                phase ^= 1u;
            }
        }
    }
    return;
drain:
    for (int s = 0; s < L::kStages; ++s)
        if (pend & (1u << s)) ptx::drain_wait(proj_bar(base, L::kFull + s), (pend_par >> s) & 1u, lim);
}

__device__ void proj_mma_role(const ProjParams& p, uint32_t base, uint32_t tmem, volatile int* abort_flag) {
    using L = ProjLayout;
    constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(L::kBM, L::kBN, false);
    const uint64_t lim = p.wait_limit_ns;
    int slot = 0;
    uint32_t phase = 0, acc_phases = 0u;  // bit i: phase of accumulator i
    int t = 0;  // tiles of this CTA
    for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++t) {
        const int ab = t & 1;
        // The epilogue has emptied this accumulator (free at first use).
        if (!ptx::mbar_wait(proj_bar(base, L::kAccEmpty + ab), ((acc_phases >> ab) & 1u) ^ 1u, abort_flag,
                            p.status, lim))
            break;
        acc_phases ^= 1u << ab;
        ptx::tc_fence_after();
        bool ok = true;
        for (int kc = 0; kc < p.k_chunks; ++kc) {
            if (!(ok = ptx::mbar_wait(proj_bar(base, L::kFull + slot), phase, abort_flag, p.status, lim))) break;
            ptx::tc_fence_after();
            const uint32_t a = base + (uint32_t)slot * L::kStageBytes;
            ptx::mma_ss_k64(tmem + 256u * (uint32_t)ab, ptx::sdesc_sw128(a, 16, 1024),
                            ptx::sdesc_sw128(a + L::kABytes, 16, 1024), kIdesc, kc > 0 ? 1u : 0u);
            ptx::mma_commit(proj_bar(base, L::kEmpty + slot));
            if (++slot == L::kStages) {
                slot = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
        ptx::mma_commit(proj_bar(base, L::kAccFull + ab));
    }
    ptx::mma_commit(proj_bar(base, L::kDrain));
    ptx::drain_wait(proj_bar(base, L::kDrain), 0u, lim);
}

__device__ void proj_epilogue_role(const ProjParams& p, uint32_t base, uint32_t tmem, int wg,
                                   volatile int* abort_flag) {
    using L = ProjLayout;
    const int warp = threadIdx.x >> 5;
    const int r = (warp & 3) * 32 + (threadIdx.x & 31);  // row of the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint64_t lim = p.wait_limit_ns;
    uint32_t acc_phases = 0u;
    int t = 0;
    for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++t) {
        const ProjUnit w = proj_decode(u, p);
        const int ab = t & 1;
        const bool ok = ptx::mbar_wait(proj_bar(base, L::kAccFull + ab), (acc_phases >> ab) & 1u, abort_flag,
                                       p.status, lim);
        if (!__all_sync(0xffffffffu, ok)) return;
        acc_phases ^= 1u << ab;
        ptx::tc_fence_after();
        const int s = w.s0 + r;
        const bool row_ok = s < p.S;
        __nv_bfloat16* yrow = p.y + ((size_t)w.b * p.S + s) * p.E;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
            ptx::tmem_ld32(tmem + lane_off + 256u * (uint32_t)ab + 128u * (uint32_t)wg + 32u * (uint32_t)c, v);
            ptx::tmem_ld_wait();
            ptx::reg_fence32(v);
            const int e0 = w.e0 + 128 * wg + 32 * c;
            if (!row_ok) continue;
#pragma unroll
            for (int g = 0; g < 4; ++g) {  // 8 features = one 16-byte store
                const int e = e0 + 8 * g;
                if (e >= p.E) break;  // E is a multiple of 8
                float f[8];
#pragma unroll
                for (int x = 0; x < 8; ++x)
                    f[x] = __uint_as_float(v[8 * g + x]) + (p.bias != nullptr ? __ldg(p.bias + e + x) : 0.f);
                uint4 o;
                o.x = ptx::pack_bf16x2(f[0], f[1]);
                o.y = ptx::pack_bf16x2(f[2], f[3]);
                o.z = ptx::pack_bf16x2(f[4], f[5]);
                o.w = ptx::pack_bf16x2(f[6], f[7]);
                *reinterpret_cast<uint4*>(yrow + e) = o;
            }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(proj_bar(base, L::kAccEmpty + ab));
    }
}

template <int D>
__global__ void __launch_bounds__(ProjLayout::kThreads, 1)
    attn_out_proj_kernel(const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_w,
                         const ProjParams p) {
    using L = ProjLayout;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < L::kStages; ++s) {
            ptx::mbar_init(proj_bar(base, L::kFull + s), 1);
            ptx::mbar_init(proj_bar(base, L::kEmpty + s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(proj_bar(base, L::kAccFull + i), 1);
            ptx::mbar_init(proj_bar(base, L::kAccEmpty + i), 8);  // one per epilogue warp
        }
        ptx::mbar_init(proj_bar(base, L::kDrain), 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
        ptx::prefetch_tensormap(&tm_o);
        ptx::prefetch_tensormap(&tm_w);
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
        if (warp == 0 && lane == 0) proj_load_role<D>(&tm_o, &tm_w, p, base, abort_flag);
        if (warp == 1 && lane == 0) proj_mma_role(p, base, tmem, abort_flag);
    } else {
        ptx::regs_inc<L::kRegsWork>();
        proj_epilogue_role(p, base, tmem, (warp - 4) >> 2, abort_flag);
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

}  // namespace attn
