// attn_proj.cu -- the output-projection entry point of libattn
// (include/attn.h): argument checks, TMA descriptors, launch.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/attn.h"
#include "common.cuh"
#include "host.h"
#include "kernel_proj.cuh"

namespace attn {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_proj_mutex;
int g_proj_ready[kMaxDevices];  // 0 not yet, 1 ready, else an ATTN_ERR code

int setup_proj_kernels() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_proj_mutex);
    if (g_proj_ready[dev] == 0) {
        const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
        const bool ok = cudaFuncSetAttribute(attn_out_proj_kernel<64>, attr, (int)ProjLayout::kDynamicSmem) ==
                            cudaSuccess &&
                        cudaFuncSetAttribute(attn_out_proj_kernel<128>, attr, (int)ProjLayout::kDynamicSmem) ==
                            cudaSuccess;
        g_proj_ready[dev] = ok ? 1 : ATTN_ERR_DEVICE;
    }
    return g_proj_ready[dev] == 1 ? ATTN_OK : g_proj_ready[dev];
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" int attn_out_proj(const void* out, const void* w, const float* bias, void* y, int B, int H,
                             int S, int D, int E, void* stream) {
    if (!out || !w || !y) return ATTN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || S < 1 || E < 1) return ATTN_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
    if (E % 8 != 0) return ATTN_ERR_UNSUPPORTED;
    if ((long long)B * H > (1ll << 30) || S > (1 << 30) || (long long)H * D > (1ll << 30)) return ATTN_ERR_UNSUPPORTED;
    const uintptr_t mis = (reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(w) |
                           reinterpret_cast<uintptr_t>(y)) & 15u;
    if (mis || (reinterpret_cast<uintptr_t>(bias) & 3u)) return ATTN_ERR_MISALIGNED;
    const size_t ob = (size_t)B * H * S * D * 2, wb = (size_t)E * H * D * 2, yb = (size_t)B * S * E * 2;
    if (host::ranges_overlap(y, yb, out, ob) || host::ranges_overlap(y, yb, w, wb) ||
        (bias && host::ranges_overlap(y, yb, bias, (size_t)E * 4)))
        return ATTN_ERR_INVALID_ARG;
    const long long m_tiles = (long long)B * ((S + 127) / 128), n_tiles = (E + 255) / 256;
    if (m_tiles * n_tiles > (1ll << 31) - 1) return ATTN_ERR_UNSUPPORTED;

    int sm_count = 0;
    unsigned int* status = nullptr;
    int device = -1;
    int rc = host::current_device(&sm_count, &status, &device);
    if (rc != ATTN_OK) return rc;
    if ((rc = setup_proj_kernels()) != ATTN_OK) return rc;

    // O as [B*H, S, D] (128-row boxes); W as [1, E, H*D] (256-row boxes).
    alignas(64) CUtensorMap to, tw;
    if (host::encode_bf16_tiles(&to, device, out, D, S, (long long)B * H) != ATTN_OK ||
        host::encode_bf16_box(&tw, device, w, H * D, E, 1, ProjLayout::kBN) != ATTN_OK)
        return ATTN_ERR_INVALID_ARG;

    ProjParams p{};
    p.B = B;
    p.H = H;
    p.S = S;
    p.E = E;
    p.m_tiles_per_batch = (S + 127) / 128;
    p.n_tiles = (int)n_tiles;
    p.num_units = (int)(m_tiles * n_tiles);
    p.k_chunks = H * D / 64;
    p.bias = bias;
    p.y = static_cast<__nv_bfloat16*>(y);
    p.status = status;
    p.wait_limit_ns = host::wait_limit_ns();
    const int grid = p.num_units < sm_count ? p.num_units : sm_count;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (D == 64)
        attn_out_proj_kernel<64><<<grid, ProjLayout::kThreads, ProjLayout::kDynamicSmem, st>>>(to, tw, p);
    else
        attn_out_proj_kernel<128><<<grid, ProjLayout::kThreads, ProjLayout::kDynamicSmem, st>>>(to, tw, p);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}
