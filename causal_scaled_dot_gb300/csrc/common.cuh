// common.cuh -- constants and the kernel parameter block shared by the
// attention kernels and their host launcher, and the Philox key schedule
// that the host precomputes for them.
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
    unsigned long long dropout_seed, dropout_offset;  // Philox key (seed) and counter word (offset)
    unsigned int philox_round_keys[20];  // dropout kernels: round r's key words at [2r], [2r + 1]
    const uint8_t* keep_bits;       // element-masked kernels: [keep_heads][S][keep_row_bytes]
    int keep_heads;                 // 1 (one mask for all heads) or Hq
    int keep_row_bytes;             // 16 per 128 keys
};

// The order in which the persistent forward kernel's CTAs take their units,
// computed on the host (attn_api.cu, fwd_schedule) and passed as a kernel
// parameter: CTA c runs units order[start[c]] .. order[start[c + 1] - 1] in
// turn.  `enabled` = 0 (more units or CTAs than the table holds) selects the
// arithmetic order of unit_of_round instead.
constexpr int kSchedMaxCtas = 160;
constexpr int kSchedMaxUnits = 4096;
struct FwdSchedule {
    int enabled;
    unsigned short start[kSchedMaxCtas + 1];
    unsigned short order[kSchedMaxUnits];
};

// The Philox4x32-10 key schedule of `seed`: round r uses key words
// (lo32(seed) + r * 0x9E3779B9, hi32(seed) + r * 0xBB67AE85) mod 2^32.  The
// same for every thread of a launch, so the host computes it once and the
// kernels read each round's words from the parameter block.
inline void philox_round_keys(unsigned long long seed, unsigned int keys[20]) {
    unsigned int k0 = (unsigned int)seed, k1 = (unsigned int)(seed >> 32);
    for (int r = 0; r < 10; ++r) {
        keys[2 * r] = k0;
        keys[2 * r + 1] = k1;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
}

}  // namespace attn
