// attn_api.cu -- the C ABI of libattn (include/attn.h): argument checks, TMA
// descriptor encoding (with a small cache of encoded maps), per-device setup,
// kernel launch, and the device status word that bounded waits report
// timeouts through.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/attn.h"
#include "common.cuh"
#include "kernel_simple.cuh"
#include "kernel_ws.cuh"
#include "fwd_schedule.h"
#include "tmap_cache.h"

// Status word: bits set by device-side waits that ran out (ptx::kStatusTimeout).
__device__ unsigned int g_attn_status;

namespace attn {
namespace {

constexpr int kVersion = 100;                       // 0.1.0
constexpr unsigned long long kWaitLimitNs = 4000000000ull;  // 4 s per wait
constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int index = -1;
    int status = ATTN_OK;  // ATTN_OK, or why this device cannot run the kernels
    int sm_count = 0;
    unsigned int* status_word = nullptr;
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

template <typename K>
cudaError_t allow_smem(K kernel, uint32_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int D, bool F, bool M, bool DR, bool E>
bool allow_ws() {
    return allow_smem(attn_fwd_ws_kernel<D, F, M, DR, E>, WsLayout<D, F>::kDynamicSmem) == cudaSuccess;
}

// Every instantiation of the persistent forward kernel that launch_any uses.
template <int D>
bool allow_ws_bf16() {
    return allow_ws<D, false, false, false, false>() && allow_ws<D, false, true, false, false>() &&
           allow_ws<D, false, false, true, false>() && allow_ws<D, false, false, false, true>() &&
           allow_ws<D, false, true, false, true>() && allow_ws<D, false, true, true, false>() &&
           allow_ws<D, false, false, true, true>() && allow_ws<D, false, true, true, true>();
}
bool allow_ws_all() {
    return allow_ws_bf16<64>() && allow_ws_bf16<128>() && allow_ws<128, true, false, false, false>() &&
           allow_ws<128, true, true, false, false>() && allow_ws<128, true, false, false, true>() &&
           allow_ws<128, true, true, false, true>();
}

// Per-device setup, once: capability check, SM count, status-word address,
// shared-memory opt-in for every kernel.  Caller holds g_mutex.
int setup_device_locked(int dev) {
    DeviceState& st = g_devices[dev];
    if (st.ready) return st.status;
    st.index = dev;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return ATTN_ERR_DEVICE;  // not cached: may be transient
    st.ready = true;
    if (major != 10 || minor != 3) {
        st.status = ATTN_ERR_UNSUPPORTED;
        return st.status;
    }
    st.sm_count = sms;
    void* word = nullptr;
    if (cudaGetSymbolAddress(&word, g_attn_status) != cudaSuccess ||
        allow_smem(attn_fwd_simple_kernel<64>, SimpleLayout<64>::kDynamicSmem) != cudaSuccess ||
        allow_smem(attn_fwd_simple_kernel<128>, SimpleLayout<128>::kDynamicSmem) != cudaSuccess ||
        !allow_ws_all()) {
        st.status = ATTN_ERR_DEVICE;
        return st.status;
    }
    st.status_word = static_cast<unsigned int*>(word);
    if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr) {
            st.status = ATTN_ERR_DEVICE;
            return st.status;
        }
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    st.status = ATTN_OK;
    return st.status;
}

int current_device_state(DeviceState** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_DEVICE;
    // A thread that has made no context-binding runtime call reports device 0
    // with no driver context current, and the tensor-map encoder is a driver
    // call that then fails; binding the device's primary context here makes
    // every entry point callable from any thread (an autograd worker, say).
    if (cudaSetDevice(dev) != cudaSuccess) return ATTN_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mutex);
    const int rc = setup_device_locked(dev);
    *out = &g_devices[dev];
    return rc;
}

// Rank-3 view [rows_outer, S, D] of a contiguous [.., S, D] tensor whose
// elements are `elem_bytes` wide, box {128 bytes of a row, box_rows, 1},
// 128-byte swizzle: one box fills box_rows rows of 128 bytes, the canonical
// K-major (and MN-major) SW128 operand layout.  Rows past S read as zero.
// Encoded maps are kept in a small cache keyed by every input of the encode
// (tmap_cache.h), so repeated calls on the same buffers skip the encoder.
std::mutex g_tmap_mutex;
TmapCache<64> g_tmap_cache;

int encode_3d(CUtensorMap* map, int device, const void* ptr, int elem_bytes, int D, int S, long long outer,
              int box_rows) {
    const TmapKey key{device, ptr, elem_bytes, D, S, outer, box_rows};
    {
        std::lock_guard<std::mutex> lock(g_tmap_mutex);
        if (g_tmap_cache.lookup(key, map)) return ATTN_OK;
    }
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)outer};
    cuuint64_t strides[2] = {(cuuint64_t)D * elem_bytes, (cuuint64_t)S * (cuuint64_t)D * elem_bytes};
    cuuint32_t box[3] = {(cuuint32_t)(128 / elem_bytes), (cuuint32_t)box_rows, 1};
    cuuint32_t elem[3] = {1, 1, 1};
    const CUtensorMapDataType type =
        elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    CUresult r = g_encode(map, type, 3, const_cast<void*>(ptr), dims, strides, box, elem,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return ATTN_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_tmap_mutex);
    g_tmap_cache.insert(key, *map);
    return ATTN_OK;
}

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

int check_args(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
               int Hkv, int S, int D, float scale, int in_elem_bytes = 2) {
    if (!q || !k || !v || !out) return ATTN_ERR_INVALID_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || S < 1) return ATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
    // Sizes that the 32-bit TMA coordinates and grid dimensions can address.
    if ((long long)B * Hq > (1ll << 30) || S > (1 << 30)) return ATTN_ERR_UNSUPPORTED;
    const uintptr_t mis = (reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                           reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out)) & 15u;
    if (mis || (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_MISALIGNED;
    const size_t q_bytes = (size_t)B * Hq * S * D * in_elem_bytes;
    const size_t kv_bytes = (size_t)B * Hkv * S * D * in_elem_bytes;
    const size_t o_bytes = (size_t)B * Hq * S * D * 2;
    if (ranges_overlap(out, o_bytes, q, q_bytes) || ranges_overlap(out, o_bytes, k, kv_bytes) ||
        ranges_overlap(out, o_bytes, v, kv_bytes))
        return ATTN_ERR_INVALID_ARG;
    if (lse) {
        const size_t l_bytes = (size_t)B * Hq * S * 4;
        if (ranges_overlap(lse, l_bytes, out, o_bytes) || ranges_overlap(lse, l_bytes, q, q_bytes) ||
            ranges_overlap(lse, l_bytes, k, kv_bytes) || ranges_overlap(lse, l_bytes, v, kv_bytes))
            return ATTN_ERR_INVALID_ARG;
    }
    return ATTN_OK;
}

// A mask input (bytes at m) may not overlap the outputs it would be read
// alongside: O (and LSE when given).
int check_mask_overlap(const void* m, size_t m_bytes, const void* out, const float* lse, int B, int Hq,
                       int S, int D) {
    if (m == nullptr) return ATTN_OK;
    if (ranges_overlap(m, m_bytes, out, (size_t)B * Hq * S * D * 2)) return ATTN_ERR_INVALID_ARG;
    if (lse != nullptr && ranges_overlap(m, m_bytes, lse, (size_t)B * Hq * S * 4)) return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

template <int D>
int launch_simple(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                  const FwdParams& p, cudaStream_t stream) {
    dim3 grid(p.B * p.Hq, p.num_q_tiles), block(128);
    if (p.num_q_tiles > 65535) return ATTN_ERR_UNSUPPORTED;
    attn_fwd_simple_kernel<D><<<grid, block, SimpleLayout<D>::kDynamicSmem, stream>>>(tq, tk, tv, p);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

// The forward kernel's unit order for a shape and CTA count (fwd_schedule.h),
// from a least-recently-used cache of 32 shapes: building one takes up to
// about 0.2 ms of host time (4096 units), a lookup well under a microsecond.
// `enabled` = 0 when the kernel keeps its arithmetic order (fewer than two
// units per CTA, or more than the table holds).
struct SchedEntry {
    int bh, nq, causal, grid;
    unsigned long long last_use;
    FwdSchedule sched;
};
std::mutex g_sched_mutex;
SchedEntry g_sched_cache[32];
unsigned long long g_sched_clock = 0;

void fwd_schedule(int bh, int nq, bool causal, int grid, FwdSchedule* out) {
    std::lock_guard<std::mutex> lock(g_sched_mutex);
    SchedEntry* victim = &g_sched_cache[0];
    for (SchedEntry& e : g_sched_cache) {
        if (e.last_use != 0 && e.bh == bh && e.nq == nq && e.causal == (int)causal && e.grid == grid) {
            e.last_use = ++g_sched_clock;
            std::memcpy(out, &e.sched, sizeof *out);
            return;
        }
        if (e.last_use < victim->last_use) victim = &e;
    }
    std::memset(&victim->sched, 0, sizeof victim->sched);
    const long long units = (long long)bh * ((nq + 1) / 2);
    victim->sched.enabled = host::fwd_schedule_wanted(units, grid) &&
                                    host::build_fwd_schedule(bh, nq, causal, grid, kSchedMaxUnits, kSchedMaxCtas,
                                                             victim->sched.start, victim->sched.order)
                                ? 1
                                : 0;
    victim->bh = bh;
    victim->nq = nq;
    victim->causal = (int)causal;
    victim->grid = grid;
    victim->last_use = ++g_sched_clock;
    std::memcpy(out, &victim->sched, sizeof *out);
}

template <int D, bool F, bool M, bool DR = false, bool E = false>
int launch_ws(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
              FwdParams p, int sm_count, cudaStream_t stream) {
    const long long npairs = (p.num_q_tiles + 1) / 2;
    const long long units = (long long)p.B * p.Hq * npairs;
    if (units > (1ll << 31) - 1) return ATTN_ERR_UNSUPPORTED;
    p.num_units = (int)units;
    const int grid = (int)(units < sm_count ? units : sm_count);
    // With a block mask the units' real costs depend on the mask, which lives
    // on the device: the cost-blind arithmetic order then spreads the unit
    // count evenly instead (a 1024-key window at B4 H16 S4096: 0.158 ms, against
    // 0.189 ms in the table's order, which expects causal costs).
    static const FwdSchedule kArithmeticOrder{};  // enabled = 0
    FwdSchedule sched;
    const FwdSchedule* order = &kArithmeticOrder;
    if (!M) {
        fwd_schedule(p.B * p.Hq, p.num_q_tiles, p.causal != 0, grid, &sched);
        order = &sched;
    }
    attn_fwd_ws_kernel<D, F, M, DR, E><<<grid, WsLayout<D, F>::kThreads, WsLayout<D, F>::kDynamicSmem, stream>>>(
        tq, tk, tv, to, p, *order);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

// The persistent kernel's instantiation for the features a call uses: block
// mask (M), dropout (DR, bf16 only) and keep bits (E).
template <int D, bool F>
int launch_any(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
               const FwdParams& p,
               int sm, cudaStream_t st, bool m, bool dr, bool e) {
    if constexpr (F) {
        if (dr) return ATTN_ERR_UNSUPPORTED;
        if (m) return e ? launch_ws<D, F, true, false, true>(tq, tk, tv, to, p, sm, st)
                        : launch_ws<D, F, true, false, false>(tq, tk, tv, to, p, sm, st);
        return e ? launch_ws<D, F, false, false, true>(tq, tk, tv, to, p, sm, st)
                 : launch_ws<D, F, false, false, false>(tq, tk, tv, to, p, sm, st);
    } else {
        if (m) {
            if (dr) return e ? launch_ws<D, F, true, true, true>(tq, tk, tv, to, p, sm, st)
                             : launch_ws<D, F, true, true, false>(tq, tk, tv, to, p, sm, st);
            return e ? launch_ws<D, F, true, false, true>(tq, tk, tv, to, p, sm, st)
                     : launch_ws<D, F, true, false, false>(tq, tk, tv, to, p, sm, st);
        }
        if (dr) return e ? launch_ws<D, F, false, true, true>(tq, tk, tv, to, p, sm, st)
                         : launch_ws<D, F, false, true, false>(tq, tk, tv, to, p, sm, st);
        return e ? launch_ws<D, F, false, false, true>(tq, tk, tv, to, p, sm, st)
                 : launch_ws<D, F, false, false, false>(tq, tk, tv, to, p, sm, st);
    }
}

// Kernel choice: the warp-specialised persistent kernel unless the environment
// variable ATTN_FWD_KERNEL=simple selects the one-tile-per-CTA kernel (kept as
// an independently scheduled implementation for cross-checks).
bool use_simple_kernel() {
    const char* v = std::getenv("ATTN_FWD_KERNEL");
    return v != nullptr && std::strcmp(v, "simple") == 0;
}

__global__ void selftest_wait_kernel(unsigned long long limit_ns, unsigned int* status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_addr(&bar), 1);
        abort_flag = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    // Nobody arrives on `bar`: phase 0 never completes and the wait must give up.
    ptx::mbar_wait(ptx::smem_addr(&bar), 0, &abort_flag, status, limit_ns);
    __syncthreads();
    if (threadIdx.x == 0) ptx::mbar_arrive(ptx::smem_addr(&bar));  // leave the barrier balanced
}

}  // namespace
}  // namespace attn

using namespace attn;

namespace attn {
namespace {
int fwd_bf16(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
             int Hkv, int S, int D, float scale, int causal, const uint8_t* block_mask,
             int mask_heads, int dropout_p8, unsigned long long seed, unsigned long long offset,
             void* stream, const uint8_t* keep_bits = nullptr, int keep_heads = 1,
             const float* descales = nullptr);
}  // namespace
}  // namespace attn

extern "C" int attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                        int Hq, int Hkv, int S, int D, float scale, int causal, void* stream) {
    return attn::fwd_bf16(q, k, v, out, lse, B, Hq, Hkv, S, D, scale, causal, nullptr, 1, 0, 0, 0,
                          stream);
}

extern "C" int attn_fwd_block_masked(const void* q, const void* k, const void* v, void* out,
                                     float* lse, int B, int Hq, int Hkv, int S, int D, float scale,
                                     int causal, const unsigned char* block_mask, int mask_heads,
                                     void* stream) {
    if (block_mask == nullptr || (mask_heads != 1 && mask_heads != Hq)) return ATTN_ERR_INVALID_ARG;
    return attn::fwd_bf16(q, k, v, out, lse, B, Hq, Hkv, S, D, scale, causal, block_mask,
                          mask_heads, 0, 0, 0, stream);
}

extern "C" int attn_fwd_elem_masked(const void* q, const void* k, const void* v, void* out,
                                    float* lse, int B, int Hq, int Hkv, int S, int D, float scale,
                                    int causal, const unsigned char* keep_bits, int keep_heads,
                                    const unsigned char* block_mask, int mask_heads, void* stream) {
    if (keep_bits == nullptr || (keep_heads != 1 && keep_heads != Hq)) return ATTN_ERR_INVALID_ARG;
    if (block_mask != nullptr && mask_heads != 1 && mask_heads != Hq) return ATTN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(keep_bits) & 15u) return ATTN_ERR_MISALIGNED;
    return attn::fwd_bf16(q, k, v, out, lse, B, Hq, Hkv, S, D, scale, causal, block_mask,
                          block_mask != nullptr ? mask_heads : 1, 0, 0, 0, stream, keep_bits,
                          keep_heads);
}

extern "C" int attn_fwd_dropout(const void* q, const void* k, const void* v, void* out, float* lse,
                                int B, int Hq, int Hkv, int S, int D, float scale, int causal,
                                float dropout_p, unsigned long long seed, unsigned long long offset,
                                void* stream) {
    if (!std::isfinite(dropout_p) || dropout_p < 0.f) return ATTN_ERR_INVALID_ARG;
    const long p8 = std::lrint((double)dropout_p * 256.0);
    if (p8 > 255) return ATTN_ERR_INVALID_ARG;
    if (p8 > 0 && offset > 0xFFFFFFFFull) return ATTN_ERR_INVALID_ARG;  // a 32-bit counter word
    return attn::fwd_bf16(q, k, v, out, lse, B, Hq, Hkv, S, D, scale, causal, nullptr, 1, (int)p8,
                          seed, offset, stream);
}

namespace attn {
namespace {
int fwd_bf16(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
             int Hkv, int S, int D, float scale, int causal, const uint8_t* block_mask,
             int mask_heads, int dropout_p8, unsigned long long seed, unsigned long long offset,
             void* stream, const uint8_t* keep_bits, int keep_heads, const float* descales) {
    // descales != nullptr: E4M3 inputs (one byte per element, D = 128) with
    // per-tensor descales {q, k, v}.
    const bool fp8 = descales != nullptr;
    int rc = check_args(q, k, v, out, lse, B, Hq, Hkv, S, D, scale, fp8 ? 1 : 2);
    if (rc != ATTN_OK) return rc;
    if (fp8) {
        for (int i = 0; i < 3; ++i)
            if (!std::isfinite(descales[i]) || !(descales[i] > 0.f)) return ATTN_ERR_INVALID_ARG;
        if (D != 128 || dropout_p8 > 0) return ATTN_ERR_UNSUPPORTED;
    }
    const size_t nt = (size_t)((S + kTile - 1) / kTile);
    if (check_mask_overlap(block_mask, (size_t)mask_heads * nt * nt, out, lse, B, Hq, S, D) != ATTN_OK ||
        check_mask_overlap(keep_bits, (size_t)keep_heads * S * 16 * nt, out, lse, B, Hq, S, D) != ATTN_OK)
        return ATTN_ERR_INVALID_ARG;
    DeviceState* dev = nullptr;
    rc = current_device_state(&dev);
    if (rc != ATTN_OK) return rc;

    alignas(64) CUtensorMap tq, tk, tv, to;
    const int eb = fp8 ? 1 : 2;
    // O (bf16 whatever the inputs) is stored by the correction warps in boxes
    // of 32 rows, one per warp.
    const int di = dev->index;
    if (encode_3d(&tq, di, q, eb, D, S, (long long)B * Hq, kTile) != ATTN_OK ||
        encode_3d(&tk, di, k, eb, D, S, (long long)B * Hkv, kTile) != ATTN_OK ||
        encode_3d(&tv, di, v, eb, D, S, (long long)B * Hkv, kTile) != ATTN_OK ||
        encode_3d(&to, di, out, 2, D, S, (long long)B * Hq, 32) != ATTN_OK)
        return ATTN_ERR_INVALID_ARG;

    FwdParams p{};
    std::memset(&p, 0, sizeof p);
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.S = S;
    p.group = Hq / Hkv;
    p.num_q_tiles = (S + kTile - 1) / kTile;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = scale * kLog2e;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.lse = lse;
    p.status = dev->status_word;
    p.wait_limit_ns = kWaitLimitNs;
    p.o_scale = 1.f;
    p.block_mask = block_mask;
    p.mask_heads = mask_heads;
    p.keep_bits = keep_bits;
    p.keep_heads = keep_heads;
    p.keep_row_bytes = 16 * p.num_q_tiles;
    if (fp8) {
        // Scores come out of the tensor core in code units: the Q and K descales
        // join the softmax scale, the V descale scales O at the end.
        p.scale_log2 = scale * descales[0] * descales[1] * kLog2e;
        p.o_scale = descales[2];
    }
    if (dropout_p8 > 0) {
        // Kept weights are scaled by 256 / (256 - p8) along with 1 / l.
        p.dropout_p8 = dropout_p8;
        p.dropout_seed = seed;
        p.dropout_offset = offset;
        philox_round_keys(seed, p.philox_round_keys);
        p.o_scale = 256.f / (float)(256 - dropout_p8);
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool m = block_mask != nullptr, dr = dropout_p8 > 0, e = keep_bits != nullptr;
    if (fp8) return launch_any<128, true>(tq, tk, tv, to, p, dev->sm_count, st, m, false, e);
    // The one-tile-per-CTA cross-check kernel covers the plain forward only.
    if (!m && !dr && !e && use_simple_kernel())
        return D == 64 ? launch_simple<64>(tq, tk, tv, p, st) : launch_simple<128>(tq, tk, tv, p, st);
    return D == 64 ? launch_any<64, false>(tq, tk, tv, to, p, dev->sm_count, st, m, dr, e)
                   : launch_any<128, false>(tq, tk, tv, to, p, dev->sm_count, st, m, dr, e);
}
}  // namespace
}  // namespace attn

extern "C" int attn_fwd_fp8(const void* q, const void* k, const void* v, float q_descale,
                            float k_descale, float v_descale, void* out, float* lse, int B, int Hq,
                            int Hkv, int S, int D, float scale, int causal, void* stream) {
    const float ds[3] = {q_descale, k_descale, v_descale};
    return attn::fwd_bf16(q, k, v, out, lse, B, Hq, Hkv, S, D, scale, causal, nullptr, 1, 0, 0, 0, stream,
                          nullptr, 1, ds);
}

extern "C" int attn_fwd_ex(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                           int Hq, int Hkv, int S, int D, float scale, int causal,
                           const attn_options_t* opts, void* stream) {
    if (opts == nullptr)
        return attn::fwd_bf16(q, k, v, out, lse, B, Hq, Hkv, S, D, scale, causal, nullptr, 1, 0, 0, 0,
                              stream);
    if (opts->input_format != ATTN_INPUT_BF16 && opts->input_format != ATTN_INPUT_E4M3)
        return ATTN_ERR_INVALID_ARG;
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
    const float ds[3] = {opts->q_descale, opts->k_descale, opts->v_descale};
    return attn::fwd_bf16(q, k, v, out, lse, B, Hq, Hkv, S, D, scale, causal, opts->block_mask,
                          opts->block_mask != nullptr ? opts->mask_heads : 1, (int)p8, opts->seed,
                          opts->offset, stream, opts->keep_bits,
                          opts->keep_bits != nullptr ? opts->keep_heads : 1,
                          opts->input_format == ATTN_INPUT_E4M3 ? ds : nullptr);
}

extern "C" int attn_sync_status(void* stream) {
    DeviceState* dev = nullptr;
    int rc = current_device_state(&dev);
    if (rc != ATTN_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return ATTN_ERR_DEVICE;
    unsigned int word = 0, zero = 0;
    if (cudaMemcpy(&word, dev->status_word, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(dev->status_word, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
        return ATTN_ERR_DEVICE;
    return (word & ptx::kStatusTimeout) ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

extern "C" int attn_selftest_wait_timeout(int limit_us, void* stream) {
    if (limit_us < 1 || limit_us > 1000000) return ATTN_ERR_INVALID_ARG;
    DeviceState* dev = nullptr;
    int rc = current_device_state(&dev);
    if (rc != ATTN_OK) return rc;
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        (unsigned long long)limit_us * 1000ull, dev->status_word);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

extern "C" const char* attn_status_string(int status) {
    switch (status) {
        case ATTN_OK: return "ATTN_OK";
        case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG: invalid argument";
        case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED: unsupported head_dim, size or device";
        case ATTN_ERR_MISALIGNED: return "ATTN_ERR_MISALIGNED: pointer not 16-byte aligned";
        case ATTN_ERR_DEVICE: return "ATTN_ERR_DEVICE: CUDA device query failed";
        case ATTN_ERR_LAUNCH: return "ATTN_ERR_LAUNCH: kernel launch failed";
        case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT: a device-side wait ran out";
        default: return "unknown attn status";
    }
}

extern "C" int attn_version(void) { return kVersion; }

extern "C" int attn_fwd_schedule(int batch_heads, int num_q_tiles, int causal, int num_ctas,
                                 unsigned short* order, unsigned short* start) {
    if (order == nullptr || start == nullptr || batch_heads <= 0 || num_q_tiles <= 0 || num_ctas <= 0)
        return ATTN_ERR_INVALID_ARG;
    if (!attn::host::fwd_schedule_wanted((long long)batch_heads * ((num_q_tiles + 1) / 2), num_ctas))
        return ATTN_ERR_UNSUPPORTED;
    return attn::host::build_fwd_schedule(batch_heads, num_q_tiles, causal != 0, num_ctas, attn::kSchedMaxUnits,
                                          attn::kSchedMaxCtas, start, order)
               ? ATTN_OK
               : ATTN_ERR_UNSUPPORTED;
}

// ---------------------------------------------------------------- shared host services
#include "host.h"

namespace attn {
namespace host {

int current_device(int* sm_count, unsigned int** status_word, int* device) {
    DeviceState* dev = nullptr;
    const int rc = current_device_state(&dev);
    if (rc != ATTN_OK) return rc;
    *sm_count = dev->sm_count;
    *status_word = dev->status_word;
    *device = dev->index;
    return ATTN_OK;
}

int encode_bf16_tiles(CUtensorMap* map, int device, const void* ptr, int D, int S, long long outer) {
    return encode_3d(map, device, ptr, 2, D, S, outer, kTile);
}

int encode_bf16_box(CUtensorMap* map, int device, const void* ptr, int D, int S, long long outer,
                    int box_rows) {
    if (box_rows < 1 || box_rows > 256) return ATTN_ERR_INVALID_ARG;
    return encode_3d(map, device, ptr, 2, D, S, outer, box_rows);
}

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
    return attn::ranges_overlap(a, na, b, nb);
}

unsigned long long wait_limit_ns() { return kWaitLimitNs; }

}  // namespace host
}  // namespace attn
