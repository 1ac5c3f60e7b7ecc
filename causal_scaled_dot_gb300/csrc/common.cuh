// common.cuh -- constants and the kernel parameter block shared by the
// attention kernels and their host launcher.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace attn {

constexpr int kTile = 128;  // query rows per tile, and key rows per key/value tile
constexpr float kLn2 = 0.693147180559945309f;
constexpr float kLog2e = 1.442695040888963407f;

// Everything a forward kernel needs besides its TMA descriptors.
struct FwdParams {
    int B, Hq, Hkv, S;
    int group;        // Hq / Hkv: query heads per key/value head
    int num_q_tiles;  // ceil(S / kTile)
    int causal;       // 1: mask keys after the query position
    float scale_log2; // scale * log2(e): scores go straight into exp2
    __nv_bfloat16* out;
    float* lse;                     // may be null
    unsigned int* status;           // device status word (timeouts)
    unsigned long long wait_limit_ns;  // bound on every mbarrier wait
    int num_units;                  // persistent kernels: total work units
    float o_scale;                  // multiplies O at the end (FP8: the V descale; else 1)
    const uint8_t* block_mask;      // null, or [mask_heads][nt][nt], nt = num_q_tiles
    int mask_heads;                 // 1 (one mask for all heads) or Hq
    int dropout_p8;                 // dropout kernels: weights dropped with probability p8 / 256
    unsigned long long dropout_seed, dropout_offset;  // Philox key
    const uint8_t* keep_bits;       // element-masked kernels: [keep_heads][S][keep_row_bytes]
    int keep_heads;                 // 1 (one mask for all heads) or Hq
    int keep_row_bytes;             // 16 per 128 keys
};

}  // namespace attn
