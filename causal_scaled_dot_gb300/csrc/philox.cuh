// philox.cuh -- Philox4x64-10 counter-based random numbers (Salmon, Moraes,
// Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011), for
// the dropout of attention weights.
#pragma once

#include <cstdint>

namespace attn {

// Ten rounds of (x0, x1, x2, x3) <- (hi(M1 x2) ^ x1 ^ k0, lo(M1 x2),
// hi(M0 x0) ^ x3 ^ k1, lo(M0 x0)), the key bumped by the Weyl constants after
// every round.
__device__ __forceinline__ void philox4x64_10(uint64_t x0, uint64_t x1, uint64_t x2, uint64_t x3,
                                              uint64_t k0, uint64_t k1, uint64_t out[4]) {
    constexpr uint64_t kM0 = 0xD2E7470EE14C6C93ull, kM1 = 0xCA5A826395121157ull;
    constexpr uint64_t kW0 = 0x9E3779B97F4A7C15ull, kW1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t hi0 = __umul64hi(kM0, x0), lo0 = kM0 * x0;
        const uint64_t hi1 = __umul64hi(kM1, x2), lo1 = kM1 * x2;
        x0 = hi1 ^ x1 ^ k0;
        x1 = lo1;
        x2 = hi0 ^ x3 ^ k1;
        x3 = lo0;
        k0 += kW0;
        k1 += kW1;
    }
    out[0] = x0;
    out[1] = x1;
    out[2] = x2;
    out[3] = x3;
}

}  // namespace attn
