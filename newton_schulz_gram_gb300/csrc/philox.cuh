// Counter-based random numbers and stochastic rounding of the Muon
// write-back (the Muon card: stochastic rounding keyed by global index),
// shared by the standalone update kernel and the fused GEMM epilogue.
//
// Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC'11): 10 rounds of two 32 x 32 -> 64-bit multiplies
// with the published multipliers and Weyl key increments.
// Element g of a write-back uses counter (g >> 3 low, g >> 3 high, step low,
// step high), key (seed low, seed high): one output (four 32-bit words)
// serves the eight elements of a block, element g taking the 16-bit half
// (g & 1) (low half first) of word (g & 7) >> 1. The bf16 result is the high
// half of (bits(w) + u). NaN stays NaN (made quiet), an infinity stays
// infinite.
#pragma once

#include <cstdint>

namespace gns {

__device__ __forceinline__ void philox4x32_10(uint32_t (&c)[4], uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t hi0 = __umulhi(0xD2511F53u, c[0]);
        const uint32_t lo0 = 0xD2511F53u * c[0];
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c[2]);
        const uint32_t lo1 = 0xCD9E8D57u * c[2];
        const uint32_t n0 = hi1 ^ c[1] ^ k0;
        const uint32_t n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0;
        c[1] = lo1;
        c[2] = n2;
        c[3] = lo0;
    }
}

// The 16-bit draw of element e (0 .. 7) of a block from its Philox output.
__device__ __forceinline__ uint32_t sr_draw(const uint32_t (&c)[4], int e) {
    return (c[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
}

__device__ __forceinline__ uint16_t sr_bf16(float w, uint32_t u16) {
    const uint32_t b = __float_as_uint(w);
    if ((b & 0x7F800000u) == 0x7F800000u)
        return static_cast<uint16_t>((b & 0x007FFFFFu) ? ((b >> 16) | 0x40u) : (b >> 16));
    return static_cast<uint16_t>((b + u16) >> 16);
}

}  // namespace gns
