// philox.cuh -- Philox4x32-10 counter-based random numbers (Salmon, Moraes,
// Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011), for
// the dropout of attention weights.  The 32-bit variant: each round is two
// 32 x 32 -> 64-bit multiplies, which the GPU does natively.
//
// Keep rule shared by the forward and both backward kernels: weight (i, j) of
// flat head bh = b*Hq + hq is kept when byte j % 16 of the block for counter
// {j / 16, i, bh, offset} under key {seed mod 2^32, seed / 2^32} is >= p8, the
// block's 16 bytes taken word 0 first, each word little-endian.
#pragma once

#include <cstdint>

namespace attn {

// Ten rounds of (x0, x1, x2, x3) <- (hi(M1 x2) ^ x1 ^ k0, lo(M1 x2),
// hi(M0 x0) ^ x3 ^ k1, lo(M0 x0)) with the key schedule given: round r uses
// (k0, k1) = (rk[2r], rk[2r + 1]), the seed's words plus r times the Weyl
// constants (philox_round_keys in common.cuh, computed once on the host and
// read from the kernel's parameter block, so the rounds need no key
// additions; measured 9 % faster for the forward with dropout than adding
// them in every round).
__device__ __forceinline__ void philox4x32_10(uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3,
                                              const unsigned int* rk, uint32_t out[4]) {
    constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = (uint64_t)kM0 * x0;
        const uint64_t p1 = (uint64_t)kM1 * x2;
        x0 = (uint32_t)(p1 >> 32) ^ x1 ^ rk[2 * r];
        x1 = (uint32_t)p1;
        x2 = (uint32_t)(p0 >> 32) ^ x3 ^ rk[2 * r + 1];
        x3 = (uint32_t)p0;
    }
    out[0] = x0;
    out[1] = x1;
    out[2] = x2;
    out[3] = x3;
}

// Keep decisions of four keys at once.  `x` holds four random bytes and `c4`
// the byte 256 - p8 (1 <= p8 <= 255) in each of its bytes: byte b of x is
// >= p8 exactly when x_b + (256 - p8) carries out of the byte.  The carry out
// of bit 7 is the majority of the two top bits and the carry into bit 7 (bit
// 7 of the sum of the low seven bits, which cannot overflow a byte); it is
// returned in bit 7 of each byte, the other bits are not meaningful.
__device__ __forceinline__ uint32_t bytes_ge(uint32_t x, uint32_t c4) {
    const uint32_t low = (x & 0x7F7F7F7Fu) + (c4 & 0x7F7F7F7Fu);
    return (x & c4) | ((x | c4) & low);
}
// A mask for a packed bf16 pair from two of those decisions: every bit of the
// low (high) half copies bit 7 of byte `b0` (`b0` + 1) of `ge`; `sel` =
// 0x9988 for bytes 0-1, 0xBBAA for bytes 2-3 (prmt with sign replication).
__device__ __forceinline__ uint32_t pair_mask(uint32_t ge, uint32_t sel) {
    uint32_t m;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(m) : "r"(ge), "r"(sel));
    return m;
}

// The 16 keep decisions of block {key_block, row, bh, offset} (bit c for key
// 16*key_block + c) under the key schedule rk; c4 as in bytes_ge.  Each word's four decisions (bit 7 of
// its bytes) are gathered into four adjacent bits by one multiply: bits 0, 8,
// 16, 24 times 2^28 + 2^21 + 2^14 + 2^7 land on bits 28-31 with no carries.
__device__ __forceinline__ uint32_t dropout_keep16(uint32_t key_block, uint32_t row, uint32_t bh, uint32_t offset,
                                                   const unsigned int* rk, uint32_t c4) {
    uint32_t r[4];
    philox4x32_10(key_block, row, bh, offset, rk, r);
    uint32_t bits = 0u;
#pragma unroll
    for (int w = 0; w < 4; ++w)
        bits |= ((((bytes_ge(r[w], c4) >> 7) & 0x01010101u) * 0x10204080u) >> 28) << (4 * w);
    return bits;
}

// 32 x 32 bit-matrix transpose across a warp: lane l holds row l (bit b =
// element (l, b)) and gets back column l (bit b = element (b, l)).  Stage j =
// 16, 8, 4, 2, 1 swaps the off-diagonal j x j blocks of every 2j x 2j block
// between lanes l and l ^ j: the lane with bit j clear keeps the columns with
// bit j clear and takes its partner's, shifted up by j; its partner keeps the
// other columns and takes the rest, shifted down.
__device__ __forceinline__ uint32_t warp_transpose_bits(uint32_t x) {
    const uint32_t lane = threadIdx.x & 31u;
    uint32_t low = 0x0000FFFFu;  // columns with bit j clear
#pragma unroll
    for (uint32_t j = 16; j > 0; j >>= 1) {
        const uint32_t y = __shfl_xor_sync(0xffffffffu, x, (int)j);
        x = (lane & j) ? (x & ~low) | ((y & ~low) >> j) : (x & low) | ((y & low) << j);
        low ^= low << (j >> 1);
    }
    return x;
}

}  // namespace attn
