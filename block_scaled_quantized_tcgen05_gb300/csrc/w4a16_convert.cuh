// w4a16_convert.cuh -- int4 x UE8M0 -> fp16 conversion used by the weight-only int4 GEMMs.
//
// A packed word holds 8 int4 weights of one row, k = 8w .. 8w + 7, even k in the low nibble of
// each byte (two's complement).  The fp16 weight is q * 2^(e - 127) with e the row's UE8M0 scale
// byte for that 32-block of k.  That product is an fp16 value for every q in -8..7 exactly when
// 103 <= e <= 139 (the fold window: 2^-24 is the smallest fp16 subnormal, 8 * 2^12 the largest
// power of two times 8 below 65504).  Output words are fp16x2 pairs in k order (low half = even k).
//
// Outside the window the converters write 0 (and NaN for the NaN code 255, since q * NaN is NaN
// for every q, zero included).  A block that holds only zero weights is then still exact; a row
// with a nonzero weight in an out-of-window block (an "outlier row", w4_row_is_outlier) is
// recomputed exactly by w4a16_outlier_kernel, which runs after the GEMM on the same stream.
#pragma once

#include <cstdint>

namespace qg {

constexpr uint32_t W4_FOLD_LO = 103;   // fold window of UE8M0 bytes, inclusive
constexpr uint32_t W4_FOLD_HI = 139;
constexpr uint32_t UE8M0_NAN = 255;

// A byte outside the fold window that is not the NaN code.
__device__ __forceinline__ bool w4_byte_outside(uint32_t e) {
    return e != UE8M0_NAN && (e - W4_FOLD_LO) > (W4_FOLD_HI - W4_FOLD_LO);
}

// True when the 32-block b of a packed int4 row (16 bytes at wrow + 16 b, 16-byte aligned) holds
// a nonzero weight.  int4 zero is the nibble 0, so the bytes are all zero exactly when every q is.
__device__ __forceinline__ bool w4_block_live(const uint8_t *wrow, int b) {
    const uint4 d = __ldg(reinterpret_cast<const uint4 *>(wrow + 16 * b));
    return (d.x | d.y | d.z | d.w) != 0u;
}

// Outlier row: some block's scale byte lies outside the fold window (and is not 255) while the
// block holds a nonzero weight.  srow: the row's nblk scale bytes; wrow: its packed weights.
// Sixteen (or four) scale bytes are tested at a time when srow is 16- (or 4-) byte aligned.
__device__ __forceinline__ uint32_t w4_outside4(uint32_t w) {
    // per byte: 0xFF where e - 103 (mod 256) > 36 and e != 255
    return __vcmpgtu4(__vsub4(w, 0x67676767u), 0x24242424u) & ~__vcmpeq4(w, 0xFFFFFFFFu);
}

__device__ __forceinline__ bool w4_row_is_outlier(const uint8_t *srow, const uint8_t *wrow,
                                                  int nblk) {
    int b = 0;
    if ((reinterpret_cast<uintptr_t>(srow) & 15u) == 0) {
        for (; b + 16 <= nblk; b += 16) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(srow + b));
            if ((w4_outside4(v.x) | w4_outside4(v.y) | w4_outside4(v.z) | w4_outside4(v.w)) == 0u)
                continue;
            const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
            for (int i = 0; i < 4; ++i) {
                const uint32_t out = w4_outside4(ws[i]);
                for (int j = 0; j < 4; ++j)
                    if (((out >> (8 * j)) & 0xFFu) && w4_block_live(wrow, b + 4 * i + j)) return true;
            }
        }
    }
    if ((reinterpret_cast<uintptr_t>(srow + b) & 3u) == 0) {
        for (; b + 4 <= nblk; b += 4) {
            const uint32_t out = w4_outside4(__ldg(reinterpret_cast<const uint32_t *>(srow + b)));
            if (out) {
                for (int j = 0; j < 4; ++j)
                    if (((out >> (8 * j)) & 0xFFu) && w4_block_live(wrow, b + j)) return true;
            }
        }
    }
    for (; b < nblk; ++b)
        if (w4_byte_outside(__ldg(srow + b)) && w4_block_live(wrow, b)) return true;
    return false;
}

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

// fp16x2 scale the general conversion multiplies by: 2^(e-127) inside the fold window
// (subnormal below 2^-14), NaN for 255, 0 for every other byte (see the file comment).
__device__ __forceinline__ uint32_t ue8m0_to_f16x2(uint32_t e) {
    uint32_t h;
    if (e == UE8M0_NAN) h = 0x7E00u;
    else if (w4_byte_outside(e)) h = 0u;
    else if (e >= 113u) h = (e - 112u) << 10;   // 2^(e-127) >= 2^-14: normal
    else h = 1u << (e - 103u);                  // 2^-24 .. 2^-15: subnormal
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
