// attn_bwd.cu -- the backward entry point of libattn (include/attn.h):
// argument checks, TMA descriptors, and the two kernel launches (dQ with
// delta, then dK/dV) on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <algorithm>
#include <mutex>

#include "../../include/attn.h"
#include "common.cuh"
#include "host.h"
#include "kernel_bwd.cuh"

namespace attn {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_bwd_mutex;
int g_bwd_ready[kMaxDevices];  // 0 not yet, 1 ready, else an ATTN_ERR code

template <typename K>
cudaError_t allow_smem(K kernel, uint32_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int D, bool M, bool E, bool DR>
bool allow_all() {
    return allow_smem(attn_bwd_dq_kernel<D, M, E, DR>, DqLayout<D>::kDynamicSmem) == cudaSuccess &&
           allow_smem(attn_bwd_dkdv_kernel<D, M, E, DR>, DkvLayout<D>::kDynamicSmem) == cudaSuccess;
}

// Every combination of block mask (M), keep bits (E) and dropout (DR).
template <int D>
bool allow_variants() {
    return allow_all<D, false, false, false>() && allow_all<D, true, false, false>() &&
           allow_all<D, false, true, false>() && allow_all<D, true, true, false>() &&
           allow_all<D, false, false, true>() && allow_all<D, true, false, true>() &&
           allow_all<D, false, true, true>() && allow_all<D, true, true, true>();
}

// Shared-memory opt-in of the backward kernels, once per device.
int setup_bwd_kernels() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_bwd_mutex);
    if (g_bwd_ready[dev] == 0) {
        const bool ok =
            allow_variants<64>() && allow_variants<128>();
        g_bwd_ready[dev] = ok ? 1 : ATTN_ERR_DEVICE;
    }
    return g_bwd_ready[dev] == 1 ? ATTN_OK : g_bwd_ready[dev];
}

int check_bwd_args(const void* q, const void* k, const void* v, const void* out, const void* dout,
                   const float* lse, float* delta, void* dq, void* dk, void* dv, int B, int Hq,
                   int Hkv, int S, int D, float scale) {
    if (!q || !k || !v || !out || !dout || !lse || !delta || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || S < 1) return ATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
    if ((long long)B * Hq > (1ll << 30) || S > (1 << 30)) return ATTN_ERR_UNSUPPORTED;
    const uintptr_t mis16 = (reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                             reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out) |
                             reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(dq) |
                             reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv)) & 15u;
    const uintptr_t mis4 = (reinterpret_cast<uintptr_t>(lse) | reinterpret_cast<uintptr_t>(delta)) & 3u;
    if (mis16 || mis4) return ATTN_ERR_MISALIGNED;
    // Outputs may overlap nothing else.
    const size_t qb = (size_t)B * Hq * S * D * 2, kb = (size_t)B * Hkv * S * D * 2, lb = (size_t)B * Hq * S * 4;
    const void* ins[6] = {q, k, v, out, dout, lse};
    const size_t in_bytes[6] = {qb, kb, kb, qb, qb, lb};
    const void* outs[4] = {dq, dk, dv, delta};
    const size_t out_bytes[4] = {qb, kb, kb, lb};
    for (int o = 0; o < 4; ++o) {
        for (int i = 0; i < 6; ++i)
            if (host::ranges_overlap(outs[o], out_bytes[o], ins[i], in_bytes[i])) return ATTN_ERR_INVALID_ARG;
        for (int o2 = o + 1; o2 < 4; ++o2)
            if (host::ranges_overlap(outs[o], out_bytes[o], outs[o2], out_bytes[o2])) return ATTN_ERR_INVALID_ARG;
    }
    return ATTN_OK;
}

template <int D, bool M, bool E, bool DR>
int launch_bwd(const CUtensorMap& tq, const CUtensorMap& tdo, const CUtensorMap& tk,
               const CUtensorMap& tv, BwdParams p, int sm_count, cudaStream_t stream) {
    const long long dq_units = (long long)p.B * p.Hq * p.num_tiles;
    const long long dkv_units = (long long)p.B * p.Hkv * p.num_tiles;
    if (dq_units > (1ll << 31) - 1) return ATTN_ERR_UNSUPPORTED;
    p.num_units = (int)dq_units;
    int grid = (int)(dq_units < sm_count ? dq_units : sm_count);
    // About eight units per CTA per head block: nearly the balance of a single
    // tile-major order, with half or less of the heads' operands live in L2.
    p.head_block = std::min(p.B * p.Hq, (8 * grid + p.num_tiles - 1) / p.num_tiles);
    attn_bwd_dq_kernel<D, M, E, DR><<<grid, DqLayout<D>::kThreads, DqLayout<D>::kDynamicSmem, stream>>>(tq, tdo, tk, tv, p);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
    p.num_units = (int)dkv_units;
    grid = (int)(dkv_units < sm_count ? dkv_units : sm_count);
    p.head_block = std::min(p.B * p.Hkv, (8 * grid + p.num_tiles - 1) / p.num_tiles);
    using KL = DkvLayout<D>;
    attn_bwd_dkdv_kernel<D, M, E, DR><<<grid, KL::kThreads, KL::kDynamicSmem, stream>>>(tq, tdo, tk, tv, p);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

// The instantiation for a block mask (m), keep bits (e) and dropout (dr).
template <int D>
int launch_variant(bool m, bool e, bool dr, const CUtensorMap& tq, const CUtensorMap& tdo,
                   const CUtensorMap& tk, const CUtensorMap& tv, const BwdParams& p, int sm_count,
                   cudaStream_t st) {
    if (dr)
        return m ? (e ? launch_bwd<D, true, true, true>(tq, tdo, tk, tv, p, sm_count, st)
                      : launch_bwd<D, true, false, true>(tq, tdo, tk, tv, p, sm_count, st))
                 : (e ? launch_bwd<D, false, true, true>(tq, tdo, tk, tv, p, sm_count, st)
                      : launch_bwd<D, false, false, true>(tq, tdo, tk, tv, p, sm_count, st));
    return m ? (e ? launch_bwd<D, true, true, false>(tq, tdo, tk, tv, p, sm_count, st)
                  : launch_bwd<D, true, false, false>(tq, tdo, tk, tv, p, sm_count, st))
             : (e ? launch_bwd<D, false, true, false>(tq, tdo, tk, tv, p, sm_count, st)
                  : launch_bwd<D, false, false, false>(tq, tdo, tk, tv, p, sm_count, st));
}

int bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
        const float* lse, float* delta, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S,
        int D, float scale, int causal, const uint8_t* block_mask, int mask_heads, void* stream,
        const uint8_t* keep_bits = nullptr, int keep_heads = 1, int dropout_p8 = 0,
        unsigned long long seed = 0, unsigned long long offset = 0);

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" int attn_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
                        const float* lse, float* delta, void* dq, void* dk, void* dv, int B, int Hq,
                        int Hkv, int S, int D, float scale, int causal, void* stream) {
    return attn::bwd(q, k, v, out, dout, lse, delta, dq, dk, dv, B, Hq, Hkv, S, D, scale, causal,
                     nullptr, 1, stream);
}

extern "C" int attn_bwd_block_masked(const void* q, const void* k, const void* v, const void* out,
                                     const void* dout, const float* lse, float* delta, void* dq,
                                     void* dk, void* dv, int B, int Hq, int Hkv, int S, int D,
                                     float scale, int causal, const unsigned char* block_mask,
                                     int mask_heads, void* stream) {
    if (block_mask == nullptr || (mask_heads != 1 && mask_heads != Hq)) return ATTN_ERR_INVALID_ARG;
    return attn::bwd(q, k, v, out, dout, lse, delta, dq, dk, dv, B, Hq, Hkv, S, D, scale, causal,
                     block_mask, mask_heads, stream);
}

extern "C" int attn_bwd_elem_masked(const void* q, const void* k, const void* v, const void* out,
                                    const void* dout, const float* lse, float* delta, void* dq,
                                    void* dk, void* dv, int B, int Hq, int Hkv, int S, int D,
                                    float scale, int causal, const unsigned char* keep_bits,
                                    int keep_heads, const unsigned char* block_mask, int mask_heads,
                                    void* stream) {
    if (keep_bits == nullptr || (keep_heads != 1 && keep_heads != Hq)) return ATTN_ERR_INVALID_ARG;
    if (block_mask != nullptr && mask_heads != 1 && mask_heads != Hq) return ATTN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(keep_bits) & 15u) return ATTN_ERR_MISALIGNED;
    return attn::bwd(q, k, v, out, dout, lse, delta, dq, dk, dv, B, Hq, Hkv, S, D, scale, causal,
                     block_mask, block_mask != nullptr ? mask_heads : 1, stream, keep_bits, keep_heads);
}

extern "C" int attn_bwd_ex(const void* q, const void* k, const void* v, const void* out,
                           const void* dout, const float* lse, float* delta, void* dq, void* dk,
                           void* dv, int B, int Hq, int Hkv, int S, int D, float scale, int causal,
                           const attn_options_t* opts, void* stream) {
    if (opts == nullptr)
        return attn::bwd(q, k, v, out, dout, lse, delta, dq, dk, dv, B, Hq, Hkv, S, D, scale, causal,
                         nullptr, 1, stream);
    if (opts->input_format != ATTN_INPUT_BF16) return ATTN_ERR_UNSUPPORTED;
    if (opts->block_mask != nullptr && opts->mask_heads != 1 && opts->mask_heads != Hq)
        return ATTN_ERR_INVALID_ARG;
    if (opts->keep_bits != nullptr) {
        if (opts->keep_heads != 1 && opts->keep_heads != Hq) return ATTN_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(opts->keep_bits) & 15u) return ATTN_ERR_MISALIGNED;
    }
    if (!std::isfinite(opts->dropout_p) || opts->dropout_p < 0.f) return ATTN_ERR_INVALID_ARG;
    const long p8 = std::lrint((double)opts->dropout_p * 256.0);
    if (p8 > 255) return ATTN_ERR_INVALID_ARG;
    if (p8 > 0 && opts->offset > 0xFFFFFFFFull) return ATTN_ERR_INVALID_ARG;  // a 32-bit counter word
    return attn::bwd(q, k, v, out, dout, lse, delta, dq, dk, dv, B, Hq, Hkv, S, D, scale, causal,
                     opts->block_mask, opts->block_mask != nullptr ? opts->mask_heads : 1, stream,
                     opts->keep_bits, opts->keep_bits != nullptr ? opts->keep_heads : 1, (int)p8,
                     opts->seed, opts->offset);
}

extern "C" int attn_bwd_dropout(const void* q, const void* k, const void* v, const void* out,
                                const void* dout, const float* lse, float* delta, void* dq, void* dk,
                                void* dv, int B, int Hq, int Hkv, int S, int D, float scale,
                                int causal, float dropout_p, unsigned long long seed,
                                unsigned long long offset, void* stream) {
    if (!std::isfinite(dropout_p) || dropout_p < 0.f) return ATTN_ERR_INVALID_ARG;
    const long p8 = std::lrint((double)dropout_p * 256.0);
    if (p8 > 255) return ATTN_ERR_INVALID_ARG;
    if (p8 > 0 && offset > 0xFFFFFFFFull) return ATTN_ERR_INVALID_ARG;  // a 32-bit counter word
    return attn::bwd(q, k, v, out, dout, lse, delta, dq, dk, dv, B, Hq, Hkv, S, D, scale, causal,
                     nullptr, 1, stream, nullptr, 1, (int)p8, seed, offset);
}

namespace attn {
namespace {

int bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
        const float* lse, float* delta, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S,
        int D, float scale, int causal, const uint8_t* block_mask, int mask_heads, void* stream,
        const uint8_t* keep_bits, int keep_heads, int dropout_p8, unsigned long long seed,
        unsigned long long offset) {
    int rc = check_bwd_args(q, k, v, out, dout, lse, delta, dq, dk, dv, B, Hq, Hkv, S, D, scale);
    if (rc != ATTN_OK) return rc;
    {  // mask inputs may not overlap the outputs
        const size_t nt = (size_t)((S + kTile - 1) / kTile);
        const size_t qb = (size_t)B * Hq * S * D * 2, kb = (size_t)B * Hkv * S * D * 2, lb = (size_t)B * Hq * S * 4;
        const void* masks[2] = {block_mask, keep_bits};
        const size_t mask_bytes[2] = {(size_t)mask_heads * nt * nt, (size_t)keep_heads * S * 16 * nt};
        for (int m = 0; m < 2; ++m)
            if (masks[m] != nullptr &&
                (host::ranges_overlap(masks[m], mask_bytes[m], dq, qb) ||
                 host::ranges_overlap(masks[m], mask_bytes[m], dk, kb) ||
                 host::ranges_overlap(masks[m], mask_bytes[m], dv, kb) ||
                 host::ranges_overlap(masks[m], mask_bytes[m], delta, lb)))
                return ATTN_ERR_INVALID_ARG;
    }
    int sm_count = 0;
    unsigned int* status = nullptr;
    int device = -1;
    rc = host::current_device(&sm_count, &status, &device);
    if (rc != ATTN_OK) return rc;
    rc = setup_bwd_kernels();
    if (rc != ATTN_OK) return rc;

    alignas(64) CUtensorMap tq, tdo, tk, tv;
    if (host::encode_bf16_tiles(&tq, device, q, D, S, (long long)B * Hq) != ATTN_OK ||
        host::encode_bf16_tiles(&tdo, device, dout, D, S, (long long)B * Hq) != ATTN_OK ||
        host::encode_bf16_tiles(&tk, device, k, D, S, (long long)B * Hkv) != ATTN_OK ||
        host::encode_bf16_tiles(&tv, device, v, D, S, (long long)B * Hkv) != ATTN_OK)
        return ATTN_ERR_INVALID_ARG;

    BwdParams p{};
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.S = S;
    p.group = Hq / Hkv;
    p.num_tiles = (S + kTile - 1) / kTile;
    p.causal = causal ? 1 : 0;
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    p.out = static_cast<const __nv_bfloat16*>(out);
    p.dout = static_cast<const __nv_bfloat16*>(dout);
    p.lse = lse;
    p.delta = delta;
    p.dq = static_cast<__nv_bfloat16*>(dq);
    p.dk = static_cast<__nv_bfloat16*>(dk);
    p.dv = static_cast<__nv_bfloat16*>(dv);
    p.status = status;
    p.wait_limit_ns = host::wait_limit_ns();
    p.block_mask = block_mask;
    p.mask_heads = mask_heads;
    p.keep_bits = keep_bits;
    p.keep_heads = keep_heads;
    p.keep_row_bytes = 16 * p.num_tiles;
    p.dropout_p8 = dropout_p8;
    p.dropout_seed = seed;
    p.dropout_offset = offset;
    philox_round_keys(seed, p.philox_round_keys);
    p.log2_keep_scale = dropout_p8 > 0 ? (float)(8.0 - std::log2((double)(256 - dropout_p8))) : 0.f;
    p.inv_keep_scale = (float)(256 - dropout_p8) / 256.f;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool m = block_mask != nullptr, e = keep_bits != nullptr, dr = dropout_p8 > 0;
    return D == 64 ? launch_variant<64>(m, e, dr, tq, tdo, tk, tv, p, sm_count, st)
                   : launch_variant<128>(m, e, dr, tq, tdo, tk, tv, p, sm_count, st);
}

}  // namespace
}  // namespace attn
