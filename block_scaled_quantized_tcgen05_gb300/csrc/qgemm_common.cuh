// qgemm_common.cuh -- device helpers shared by the tcgen05 GEMM kernels: tile order and the
// TMEM -> fp16 epilogue.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

#include "qgemm_ptx.cuh"

namespace qg {

// Persistent tile order.  Tiles are walked in groups of GROUP_M row-blocks: inside a group the
// row-block index changes fastest, so the CTAs running at the same time share a small set of
// A row panels and B column panels in L2 (grid-level rasterisation, the GB300 analogue of the
// block swizzle the TileLang backend applies).
constexpr int GROUP_M = 16;

__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int &mb, int &nb) {
    const int per_group = GROUP_M * tiles_n;
    const int group = t / per_group;
    const int first_m = group * GROUP_M;
    const int gsize = min(GROUP_M, tiles_m - first_m);
    const int r = t - group * per_group;
    mb = first_m + r % gsize;
    nb = r / gsize;
}

__device__ __forceinline__ uint8_t *align_1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Write 32 consecutive fp32 accumulators of one output row as fp16 to crow[col0 .. col0 + 31],
// masking columns >= N.  `vec` says crow + col0 is 16-byte aligned (C 16-byte aligned and its
// row stride a multiple of 8 elements); otherwise 2-byte stores are used.
__device__ __forceinline__ void store_row_chunk32(__half *crow, int col0, int N, bool vec,
                                                  const uint32_t (&v)[32]) {
    uint32_t p[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) p[i] = pack_f16x2(__uint_as_float(v[2 * i]),
                                                   __uint_as_float(v[2 * i + 1]));
    if (vec && col0 + 32 <= N) {
        uint4 *dst = reinterpret_cast<uint4 *>(crow + col0);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2],
                                                        p[4 * i + 3]);
    } else {
        uint16_t *dst = reinterpret_cast<uint16_t *>(crow + col0);
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (col0 + i < N) dst[i] = static_cast<uint16_t>((p[i >> 1] >> ((i & 1) * 16)) & 0xFFFF);
    }
}

}  // namespace qg
