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

// Work items of a persistent CTA-pair kernel: whole tiles, then -- when the tiles left after the
// last full wave of pairs fit twice into one wave -- each leftover tile as two column halves, so
// the last wave takes half a tile's time instead of a whole one.  half < 0 marks a whole tile.
// A column of the product does not depend on the other columns, so the split leaves every output
// bit unchanged.
struct PairWork {
    int full_items, n_items;
    __device__ __forceinline__ PairWork(int num_tiles, int npairs) {
        const int rem = num_tiles % npairs;
        const bool split = rem > 0 && 2 * rem <= npairs;
        full_items = num_tiles - (split ? rem : 0);
        n_items = full_items + (split ? 2 * rem : 0);
    }
    __device__ __forceinline__ void item(int it, int &tile, int &half) const {
        if (it < full_items) {
            tile = it;
            half = -1;
        } else {
            tile = full_items + ((it - full_items) >> 1);
            half = (it - full_items) & 1;
        }
    }
};

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
        for (int i = 0; i < 4; ++i)
            st_global_stream(dst + i, make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]));
    } else {
        uint16_t *dst = reinterpret_cast<uint16_t *>(crow + col0);
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (col0 + i < N) dst[i] = static_cast<uint16_t>((p[i >> 1] >> ((i & 1) * 16)) & 0xFFFF);
    }
}

// Epilogue flags, as EPI_* on the host: bit 0 adds the existing output, bit 1 applies ReLU.
constexpr int EPI_ACC_BIT = 1;
constexpr int EPI_RELU_BIT = 2;

// The fused epilogue on 32 fp32 accumulators of one output row (columns col0 .. col0 + 31 of
// crow): x = acc (+ fp32(C_old) when accumulating, C_old read before it is overwritten), then
// max(x, +0) for ReLU.  Columns >= N are not read.
__device__ __forceinline__ void epilogue_math32(uint32_t (&v)[32], const __half *crow, int col0,
                                                int N, bool vec, int epi) {
    if (epi & EPI_ACC_BIT) {
        if (vec && col0 + 32 <= N) {
            const uint4 *src = reinterpret_cast<const uint4 *>(crow + col0);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 w = src[i];
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const __half2 h = *reinterpret_cast<const __half2 *>(&ww[j]);
                    v[8 * i + 2 * j] = __float_as_uint(__uint_as_float(v[8 * i + 2 * j]) + __low2float(h));
                    v[8 * i + 2 * j + 1] =
                        __float_as_uint(__uint_as_float(v[8 * i + 2 * j + 1]) + __high2float(h));
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (col0 + i < N)
                    v[i] = __float_as_uint(__uint_as_float(v[i]) + __half2float(crow[col0 + i]));
        }
    }
    if (epi & EPI_RELU_BIT) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(fmaxf(__uint_as_float(v[i]), 0.0f));
    }
}

// Drain one 128 x BN fp32 accumulator tile to fp16 global memory.  The warp reads its TMEM lane
// quarter q (rows 32 q .. 32 q + 31 of the tile, one row per lane) 32 columns at a time.
// Direct form: each lane stores its own row (16-byte stores).  Staged form (`stage` = 2 KB of
// shared memory owned by this warp): the 32 x 32 fp16 chunk goes through shared memory (16-byte
// chunks swizzled by row pair, conflict-free both ways) so that each store instruction writes
// 8 rows x 64 contiguous bytes, i.e. whole 32-byte sectors.  The accumulator is released
// (arrival on `tmem_empty`) after its last column has been read.
// `epi` (EPI_ACC_BIT | EPI_RELU_BIT) fuses C = relu?(acc [+ C_old]) before the fp16 rounding.
// RELEASE selects how the accumulator is released: 0 = every lane arrives on this CTA's barrier;
// 2 = one lane per warp arrives on `tmem_empty` given as a shared::cluster address (a CTA pair
// releases its accumulators on the MMA-issuing CTA's barrier) with cluster-scope release
// semantics; 3 = the same arrival relaxed (the TMEM reads it covers are complete at
// tcgen05.wait::ld, so no memory ordering is needed, and a cluster-scope release costs about a
// microsecond).
template <int BN, int RELEASE = 0>
__device__ __forceinline__ void epilogue_tile(uint32_t tmem_base, uint32_t q, uint32_t lane,
                                              __half *C, int64_t ldc, int m0, int n0, int M,
                                              int N, bool vec, uint32_t tmem_empty,
                                              uint32_t stage, int epi = 0) {
    const int row = m0 + static_cast<int>(q * 32 + lane);
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ++ch) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_base + ((q * 32) << 16) + ch * 32, v);
        tmem_wait_ld();
        if (ch == BN / 32 - 1) {
            tc_fence_before();
            if constexpr (RELEASE == 2) {
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tmem_empty);
            } else if constexpr (RELEASE == 3) {
                __syncwarp();
                if (lane == 0) mbar_arrive_relaxed_cluster(tmem_empty);
            } else {
                mbar_arrive(tmem_empty);
            }
        }
        const int col0 = n0 + ch * 32;
        if (epi != 0 && row < M) epilogue_math32(v, C + static_cast<int64_t>(row) * ldc, col0, N, vec, epi);
        if (stage == 0u || !vec) {
            if (row < M) store_row_chunk32(C + static_cast<int64_t>(row) * ldc, col0, N, vec, v);
            continue;
        }
        uint32_t p[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            p[i] = pack_f16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
        const uint32_t sw = (lane >> 1) & 3;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t a = stage + lane * 64 + ((j ^ sw) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(p[4 * j]),
                         "r"(p[4 * j + 1]), "r"(p[4 * j + 2]), "r"(p[4 * j + 3])
                         : "memory");
        }
        __syncwarp();
        const uint32_t c16 = lane & 3;           // 16-byte chunk of the row this lane stores
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t r = (lane >> 2) + 8 * i;                    // row within the 32
            uint4 w;
            const uint32_t a = stage + r * 64 + ((c16 ^ ((r >> 1) & 3)) << 4);
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                         : "r"(a)
                         : "memory");
            const int grow = m0 + static_cast<int>(q * 32 + r);
            const int gcol = col0 + static_cast<int>(8 * c16);
            if (grow < M) {
                __half *dst = C + static_cast<int64_t>(grow) * ldc + gcol;
                if (gcol + 8 <= N) {
                    st_global_stream(dst, w);
                } else {
                    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (gcol + e < N)
                            reinterpret_cast<uint16_t *>(dst)[e] =
                                static_cast<uint16_t>((ww[e >> 1] >> ((e & 1) * 16)) & 0xFFFF);
                }
            }
        }
        __syncwarp();
    }
}

// Split-K: drain one 128 x BN fp32 accumulator tile, unrounded, into a partial plane P (row
// stride ldp floats, rows 16-byte aligned, every column of the tile inside a row).  The warp's 32
// rows go through its 2 KB of shared memory 16 columns at a time (the row-pair swizzle of the fp16
// staging above), so each store instruction writes 8 rows x 64 contiguous bytes.  Rows >= M are
// not written.  The accumulator is released (every lane arrives on `tmem_empty`) after its last
// column has been read.
template <int BN>
__device__ __forceinline__ void partial_tile(uint32_t tmem_base, uint32_t q, uint32_t lane,
                                             float *P, int64_t ldp, int m0, int n0, int M,
                                             uint32_t tmem_empty, uint32_t stage) {
    const uint32_t sw = (lane >> 1) & 3;
    const uint32_t c16 = lane & 3;
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ++ch) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_base + ((q * 32) << 16) + ch * 32, v);
        tmem_wait_ld();
        if (ch == BN / 32 - 1) {
            tc_fence_before();
            mbar_arrive(tmem_empty);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t a = stage + lane * 64 + ((j ^ sw) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a),
                             "r"(v[16 * h + 4 * j]), "r"(v[16 * h + 4 * j + 1]),
                             "r"(v[16 * h + 4 * j + 2]), "r"(v[16 * h + 4 * j + 3])
                             : "memory");
            }
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t r = (lane >> 2) + 8 * i;
                uint4 w;
                const uint32_t a = stage + r * 64 + ((c16 ^ ((r >> 1) & 3)) << 4);
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                             : "r"(a)
                             : "memory");
                const int grow = m0 + static_cast<int>(q * 32 + r);
                const int gcol = n0 + ch * 32 + 16 * h + static_cast<int>(4 * c16);
                if (grow < M)
                    *reinterpret_cast<uint4 *>(P + static_cast<int64_t>(grow) * ldp + gcol) = w;
            }
            __syncwarp();
        }
    }
}

// K range of split-K work item `it` of a one-CTA GEMM: tile it % num_tiles, split it / num_tiles.
// The KT k-tiles are cut into `splits` ranges of whole units of `unit` k-tiles, as even as they
// go (the first KU % splits ranges one unit longer), so a range starts on a unit boundary; the
// last unit may be short.  splits <= ceil(KT / unit) keeps every range non-empty.
__device__ __forceinline__ void split_item(int it, int num_tiles, int splits, int KT, int unit,
                                           int &tile, int &split, int &kt0, int &kt1) {
    tile = it % num_tiles;
    split = it / num_tiles;
    const int KU = (KT + unit - 1) / unit;
    const int u0 = split * (KU / splits) + min(split, KU % splits);
    const int u1 = u0 + KU / splits + (split < KU % splits ? 1 : 0);
    kt0 = unit * u0;
    kt1 = min(KT, unit * u1);
}

// Stage one 32 x 32 fp16 chunk (16 packed pairs per lane, lane = row) through this warp's 2 KB of
// shared memory and store it with whole-sector 16-byte stores (rows >= M and columns >= N masked).
__device__ __forceinline__ void store_chunk_staged(const uint32_t (&p)[16], uint32_t lane,
                                                   uint32_t stage, __half *C, int64_t ldc,
                                                   int row0, int col0, int M, int N) {
    const uint32_t sw = (lane >> 1) & 3;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t a = stage + lane * 64 + ((j ^ sw) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(p[4 * j]),
                     "r"(p[4 * j + 1]), "r"(p[4 * j + 2]), "r"(p[4 * j + 3])
                     : "memory");
    }
    __syncwarp();
    const uint32_t c16 = lane & 3;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t r = (lane >> 2) + 8 * i;
        uint4 w;
        const uint32_t a = stage + r * 64 + ((c16 ^ ((r >> 1) & 3)) << 4);
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                     : "r"(a)
                     : "memory");
        const int grow = row0 + static_cast<int>(r);
        const int gcol = col0 + static_cast<int>(8 * c16);
        if (grow < M) {
            __half *dst = C + static_cast<int64_t>(grow) * ldc + gcol;
            if (gcol + 8 <= N) {
                st_global_stream(dst, w);
            } else {
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (gcol + e < N)
                        reinterpret_cast<uint16_t *>(dst)[e] =
                            static_cast<uint16_t>((ww[e >> 1] >> ((e & 1) * 16)) & 0xFFFF);
            }
        }
    }
    __syncwarp();
}

// As epilogue_tile (staged form; `vec` must hold), software-pipelined: the TMEM read of chunk c + 1
// is issued before chunk c is stored, so TMEM latency overlaps the stores and the accumulator is
// released as soon as the last chunk has been read.
template <int BN, int RELEASE = 0>
__device__ __forceinline__ void epilogue_tile_pipelined(uint32_t tmem_base, uint32_t q,
                                                        uint32_t lane, __half *C, int64_t ldc,
                                                        int m0, int n0, int M, int N,
                                                        uint32_t tmem_empty, uint32_t stage) {
    constexpr int NCH = BN / 32;
    const uint32_t taddr = tmem_base + ((q * 32) << 16);
    const int row0 = m0 + static_cast<int>(q * 32);
    uint32_t v[32];
    tmem_ld_32x32b_x32(taddr, v);
#pragma unroll 1
    for (int ch = 0; ch < NCH; ++ch) {
        tmem_wait_ld();
        uint32_t p[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            p[i] = pack_f16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
        if (ch + 1 < NCH) {
            tmem_ld_32x32b_x32(taddr + (ch + 1) * 32, v);
        } else {
            tc_fence_before();
            if constexpr (RELEASE == 2) {
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tmem_empty);
            } else {
                mbar_arrive(tmem_empty);
            }
        }
        store_chunk_staged(p, lane, stage, C, ldc, row0, n0 + ch * 32, M, N);
    }
}

// Store 16 packed fp16 pairs (32 columns of one output row) to crow[col0 .. col0 + 31], masking
// columns >= N; 16-byte streaming stores when `vec` (see store_row_chunk32).
__device__ __forceinline__ void store_row_packed16(__half *crow, int col0, int N, bool vec,
                                                   const uint32_t (&p)[16]) {
    if (vec && col0 + 32 <= N) {
        uint4 *dst = reinterpret_cast<uint4 *>(crow + col0);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            st_global_stream(dst + i, make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]));
    } else {
        uint16_t *dst = reinterpret_cast<uint16_t *>(crow + col0);
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (col0 + i < N) dst[i] = static_cast<uint16_t>((p[i >> 1] >> ((i & 1) * 16)) & 0xFFFF);
    }
}

// As epilogue_tile, but the warp's whole 32 x BN slice is read from TMEM (16 columns at a time)
// and packed to fp16 in registers (BN / 32 x 16 of them) before anything is stored, and the accumulator is released
// right after the reads: the next tile's MMAs wait for the TMEM reads only, while the stores run
// under them.  Release as RELEASE = 3 of epilogue_tile (one relaxed arrival per warp on
// `tmem_empty`, a shared::cluster address).  `relu` applies max(x, +0) before the rounding; the
// accumulate epilogue (which reads the old C) takes epilogue_tile.
template <int BN>
__device__ __forceinline__ void epilogue_tile_early(uint32_t tmem_base, uint32_t q, uint32_t lane,
                                                    __half *C, int64_t ldc, int m0, int n0, int M,
                                                    int N, bool vec, uint32_t tmem_empty,
                                                    uint32_t stage, bool relu = false) {
    constexpr int NCH = BN / 32;
    uint32_t p[NCH][16];
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {      // 32 columns per read: one wait per 32 (each wait
        uint32_t v[32];                     // covers every load in flight, so fewer is faster)
        tmem_ld_32x32b_x32(tmem_base + ((q * 32) << 16) + ch * 32, v);
        tmem_wait_ld();
        if (relu) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(fmaxf(__uint_as_float(v[i]), 0.0f));
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
            p[ch][i] = pack_f16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive_relaxed_cluster(tmem_empty);
    const int row = m0 + static_cast<int>(q * 32 + lane);
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
        const int col0 = n0 + ch * 32;
        if (stage == 0u || !vec) {
            if (row < M) store_row_packed16(C + static_cast<int64_t>(row) * ldc, col0, N, vec, p[ch]);
            continue;
        }
        // 32 x 32 chunk through this warp's 2 KB of shared memory (16-byte chunks swizzled by row
        // pair), then 8 rows x 64 contiguous bytes per store instruction
        const uint32_t sw = (lane >> 1) & 3;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t a = stage + lane * 64 + ((j ^ sw) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(p[ch][4 * j]),
                         "r"(p[ch][4 * j + 1]), "r"(p[ch][4 * j + 2]), "r"(p[ch][4 * j + 3])
                         : "memory");
        }
        __syncwarp();
        const uint32_t c16 = lane & 3;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t r = (lane >> 2) + 8 * i;
            uint4 w;
            const uint32_t a = stage + r * 64 + ((c16 ^ ((r >> 1) & 3)) << 4);
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                         : "r"(a)
                         : "memory");
            const int grow = m0 + static_cast<int>(q * 32 + r);
            const int gcol = col0 + static_cast<int>(8 * c16);
            if (grow < M) {
                __half *dst = C + static_cast<int64_t>(grow) * ldc + gcol;
                if (gcol + 8 <= N) {
                    st_global_stream(dst, w);
                } else {
                    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (gcol + e < N)
                            reinterpret_cast<uint16_t *>(dst)[e] =
                                static_cast<uint16_t>((ww[e >> 1] >> ((e & 1) * 16)) & 0xFFFF);
                }
            }
        }
        __syncwarp();
    }
}

}  // namespace qg
