// w4a16_convert.cuh -- int4 x UE8M0 -> fp16 conversion used by the weight-only int4 GEMMs.
//
// A packed word holds 8 int4 weights of one row, k = 8w .. 8w + 7, even k in the low nibble of
// each byte (two's complement).  The fp16 weight is q * 2^(e - 127) with e the row's UE8M0 scale
// byte for that 32-block of k; it is exact for 103 <= e <= 139 (fp16 normal and subnormal range
// for |q| <= 8).  Output words are fp16x2 pairs in k order (low half = even k).
#pragma once

#include <cstdint>

namespace qg {

__device__ __forceinline__ uint32_t h2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}
__device__ __forceinline__ uint32_t h2_mul(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// fp16 bits of 2^(e-127) for e in [103, 142] (subnormals below 2^-14); outside that range the
// nearest representable behaviour: 0 below, +inf above.
__device__ __forceinline__ uint32_t ue8m0_to_f16x2(uint32_t e) {
    const int x = static_cast<int>(e) - 127;
    uint32_t h;
    if (x > 15) h = 0x7C00u;
    else if (x >= -14) h = static_cast<uint32_t>(x + 15) << 10;
    else if (x >= -24) h = 1u << (x + 24);
    else h = 0u;
    return h | (h << 16);
}

// Fused path, exact for scale exponents x = e - 127 in [-10, 5]: byte j of the biased word is
// spread to both halves, the low nibble as 1024 + u and the high nibble as 1024 + 16 u, and one
// fp16x2 FMA with per-half constants (s, s/16) and (-1032 s, -72 s) gives (q_lo s, q_hi s).
__device__ __forceinline__ bool fused_ok(uint32_t e) { return e >= 117u && e <= 132u; }

__device__ __forceinline__ void fused_consts(uint32_t e, uint32_t &s2, uint32_t &c2) {
    const uint32_t x15 = e - 112u;                          // x + 15
    const uint32_t s = x15 << 10, s16 = (x15 - 4u) << 10;   // 2^x, 2^(x-4)
    const uint32_t c1032 = 0x8000u | ((x15 + 10u) << 10) | 8u;    // -1032 * 2^x
    const uint32_t c72 = 0x8000u | ((x15 + 6u) << 10) | 128u;     // -72 * 2^x
    s2 = s | (s16 << 16);
    c2 = c1032 | (c72 << 16);
}

// The +8 bias (the nibble's sign bit flipped) and the 1024 exponent go in with one lop3,
// (b & 0x00F0000F) ^ 0x64806408: inside the mask it flips bit 3 of each kept nibble, outside it
// writes the exponent bits.
__device__ __forceinline__ void i4x8_to_f16_fused(uint32_t v, uint32_t s2, uint32_t c2,
                                                  uint32_t (&o)[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t b = __byte_perm(v, 0u, 0x4040u | (j << 8) | j);   // byte j in both halves
        uint32_t tv;
        asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(tv) : "r"(b), "r"(0x00F0000Fu), "r"(0x64806408u));
        o[j] = h2_fma(tv, s2, c2);
    }
}

// 8 int4 (one 32-bit word, k = 8w .. 8w+7, even k in low nibbles) times the fp16x2 scale ->
// four fp16x2 words in k order.  Each pair comes out of the same spread as the fused path; one
// fp16x2 FMA with per-half constants (1, 1/16) and (-1032, -72) gives the exact (q_lo, q_hi),
// and the multiply by the scale is the one rounding.
__device__ __forceinline__ void i4x8_to_f16(uint32_t v, uint32_t s2, uint32_t (&o)[4]) {
    const uint32_t ONE_R16 = 0x2C003C00u;   // (1, 1/16)
    const uint32_t BIAS = 0xD480E408u;      // (-1032, -72)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t b = __byte_perm(v, 0u, 0x4040u | (j << 8) | j);   // byte j in both halves
        uint32_t tv;
        asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(tv) : "r"(b), "r"(0x00F0000Fu), "r"(0x64806408u));
        o[j] = h2_mul(h2_fma(tv, ONE_R16, BIAS), s2);
    }
}

}  // namespace qg
