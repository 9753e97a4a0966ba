// mxfp8_gemm.cu -- block-scaled FP8 (E4M3 data, UE8M0 scale per 32 along K) GEMM on tcgen05.
//
// C[M, N] = fp16_rn( sum_k e4m3(A[m,k]) 2^(SA[m,k/32]-127) * e4m3(B[n,k]) 2^(SB[n,k/32]-127) )
//
// The quantized matmul2d of "Optimize custom machine learning operations with Metal tensors"
// (sections "Shader MXFP8 tensor types", "Slicing and quantized matmul") re-designed for
// sm_103a: the tensor core consumes the E4M3 planes and the UE8M0 planes directly
// (tcgen05.mma kind::mxf8f6f4 with block_scale), so no dequantised copy ever exists.
//
// One persistent CTA per SM walks output tiles of 128 x BN (BN = 256, or 128 for narrow N); with
// few tiles (M or N small: a decode-sized batch) its work items are (tile, k range) pairs, each
// range's unrounded sum going to an fp32 partial plane that splitk_reduce.cu adds in order.  Two
// TMEM accumulators are used when they fit beside the per-stage scale columns (BN = 128); at
// BN = 256 the 512 TMEM columns hold one accumulator plus the scale slots.  Warp roles:
//   warp 0     producer: TMA loads of the A / B k-tiles (128 B of K per row, 128-byte swizzle)
//              and of their scale bytes, which it lays out per k-tile in the 32-line x 16-byte
//              form that tcgen05.cp.32x128b.warpx4 copies into TMEM (line i, word c = row
//              32 c + i of a 128-row group).
//   warp 1     TMEM owner and MMA issuer: per k-tile it copies the scale bytes into TMEM,
//              then issues four 128 x BN x 32 block-scaled MMAs (scale-factor id = K step).
//   warps 2-5  epilogue: TMEM -> registers -> fp16 (round to nearest even) -> global.
// Scale bytes reach shared memory by one of three routes, chosen from the scale planes'
// alignment: SFM_TMA (16-byte aligned rows: one 32-byte x rows TMA box per 8 k-tiles into one
// staging slot, read into registers at once so the next group can land, then rearranged),
// SFM_CPASYNC (4-byte aligned: 4-byte cp.async per row and k-tile), SFM_BYTES (any alignment:
// byte loads).  The epilogue stages each 32 x 32 chunk in shared memory for sector-wide stores.
// Every wait is bounded.
#include "qgemm_common.cuh"
#include "qgemm_debug.cuh"
#include "qgemm_internal.h"
#include "qgemm_ptx.cuh"

#include <algorithm>

namespace {

using namespace qg;

constexpr int BM = 128;
constexpr int BK = 128;                     // E4M3 elements (= bytes) per k-tile
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;          // 2 accumulators of BN columns + scale slots
constexpr uint32_t SF_COLS_PER_STAGE = 16;  // SFA: 4 columns, SFB: 4 per 128 rows of B
constexpr int SF_GROUP = 8;                 // k-tiles per scale group (SFM_TMA)
constexpr uint32_t SF_ROW = SF_GROUP * 4;   // bytes of one row's scales per group (32)
// Split-K ranges start on multiples of 4 k-tiles: 16 scale bytes, the TMA box's start rule.
constexpr int SPLIT_UNIT = 4;

enum { SFM_BYTES = 0, SFM_CPASYNC = 1, SFM_TMA = 2 };

template <int BN>
struct Cfg {
    static constexpr int STAGES = (BN > 128) ? 4 : 6;
    static constexpr int SFB_GROUPS = (BN + 127) / 128;   // 128-row scale groups of B
    // two accumulators when they fit beside the scale columns (BN = 224: 448 + 64 = 512)
    static constexpr int ACC_BUFS = (2 * BN + STAGES * SF_COLS_PER_STAGE <= TMEM_COLS) ? 2 : 1;
    static constexpr uint32_t SF_COL0 = ACC_BUFS * BN;   // first scale-factor TMEM column
    static constexpr uint32_t A_BYTES = BM * BK;
    static constexpr uint32_t B_BYTES = BN * BK;
    static constexpr uint32_t SFA_BYTES = BM * 4;
    static constexpr uint32_t SFB_BYTES = SFB_GROUPS * 512;
    static constexpr uint32_t STG_A = BM * SF_ROW;  // one scale group of A
    static constexpr uint32_t STG_B = SFB_GROUPS * 128 * SF_ROW;
    static constexpr uint32_t OFF_A = 0;
    static constexpr uint32_t OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr uint32_t OFF_SFA = OFF_B + STAGES * B_BYTES;
    static constexpr uint32_t OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
    static constexpr uint32_t OFF_STG = OFF_SFB + STAGES * SFB_BYTES;   // STG_A + STG_B
    static constexpr uint32_t OFF_EPI = OFF_STG + STG_A + STG_B;         // 4 warps x 2 KB
    static constexpr uint32_t OFF_BAR = OFF_EPI + 4 * 2048;
    // full[S], empty[S], tmem_full[2], tmem_empty[2], drain, sf_full, then the TMEM slot
    static constexpr uint32_t OFF_SLOT = OFF_BAR + (2 * STAGES + 6) * 8;
    static constexpr uint32_t SMEM_BYTES = OFF_SLOT + 16 + 1024;
    static_assert(SF_COL0 + STAGES * SF_COLS_PER_STAGE <= TMEM_COLS, "TMEM budget");
    static_assert(BN == 128 || BN == 224 || BN == 256, "BN");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// Instruction descriptor, kind::mxf8f6f4: A, B E4M3 (format 0), K-major, D fp32 (implicit),
// N >> 3 at bit 17, scale type UE8M0 (bit 23), M >> 7 at bit 27.  The K-step selects which
// byte of each 32-bit TMEM scale word is used: A's id at bits 29-30, B's at bits 4-5.
__host__ __device__ constexpr uint32_t mx_idesc(int n) {
    return (static_cast<uint32_t>(n >> 3) << 17) | (1u << 23) | (static_cast<uint32_t>(BM >> 7) << 27);
}

// Up to 4 consecutive scale bytes (little-endian in one word), zero beyond `n`.
__device__ __forceinline__ uint32_t load_scale_word(const uint8_t *p, uint32_t n) {
    uint32_t w = 0;
#pragma unroll
    for (uint32_t i = 0; i < 4; ++i)
        if (i < n) w |= static_cast<uint32_t>(__ldg(p + i)) << (8 * i);
    return w;
}

__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ uint32_t word_of(const uint4 &v, int j) {
    return j == 0 ? v.x : (j == 1 ? v.y : (j == 2 ? v.z : v.w));
}

template <int BN, int SFM>
__global__ void __launch_bounds__(THREADS, 1)
mxfp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                  const uint8_t *__restrict__ sfa, int64_t lds_a, const uint8_t *__restrict__ sfb,
                  int64_t lds_b, __half *__restrict__ C, int64_t ldc, int c_vec, int M, int N, int K,
                  int splits, float *__restrict__ P, int64_t ldp, int epi, unsigned *err,
                  uint64_t timeout_ns) {
    using G = Cfg<BN>;
    constexpr int S = G::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_1024(smem_raw);
    const uint32_t sb = smem_u32(smem);
    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    // a split-K reduction launched as a programmatic dependent may be scheduled now (it waits
    // for this grid to complete before it reads anything)
    griddep_launch_dependents();

    auto full_bar = [&](int s) { return sb + G::OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sb + G::OFF_BAR + 8u * (S + s); };
    // accumulator double buffer: tmem_full[2], tmem_empty[2], then the drain barrier
    const uint32_t acc_bar0 = sb + G::OFF_BAR + 8u * (2 * S);
    auto tmem_full = [&](uint32_t b) { return acc_bar0 + 8u * b; };
    auto tmem_empty = [&](uint32_t b) { return acc_bar0 + 16u + 8u * b; };
    const uint32_t drain_bar = acc_bar0 + 32;
    const uint32_t sf_full = acc_bar0 + 40;
    volatile uint32_t *slot = reinterpret_cast<volatile uint32_t *>(smem + G::OFF_SLOT);

    const int tiles_m = (M + BM - 1) / BM;
    const int tiles_n = (N + BN - 1) / BN;
    const int num_tiles = tiles_m * tiles_n;
    const int num_items = num_tiles * splits;        // (tile, k range) work items
    const int KT = (K + BK - 1) / BK;
    const int nkb = K / 32;                          // scale blocks per row
    const int64_t plane = static_cast<int64_t>(M) * ldp;   // floats per split-K partial plane

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1 + 32);  // producer's expect_tx arrival + 32 scale arrivals
            mbar_init(empty_bar(s), 1);      // tcgen05.commit
        }
        mbar_init(tmem_full(0), 1);
        mbar_init(tmem_full(1), 1);
        mbar_init(tmem_empty(0), 128);             // every epilogue thread
        mbar_init(tmem_empty(1), 128);
        mbar_init(drain_bar, 1);
        mbar_init(sf_full, 1);
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if constexpr (SFM == SFM_TMA) {
            tma_prefetch_desc(&tmSA);
            tma_prefetch_desc(&tmSB);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(const_cast<uint32_t *>(slot)), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *slot;

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        int issued = 0;
        int sf_issued = 0;       // scale groups requested (SFM_TMA), in CTA-local sequence (lane 0)
        int sf_waited = 0;       // scale groups whose arrival this warp has observed
        int sf_seq = 0;          // scale groups consumed
        bool ok = true;
        // The next scale group to request (lane 0): group sf_g of work item sf_it, eight k-tiles
        // from the item's first; the staging slot's barrier completes phase q when the q-th
        // request lands.
        int sf_it = static_cast<int>(blockIdx.x), sf_g = 0;
        auto issue_sf = [&]() {
            if (sf_it >= num_items) return;
            int tile, split, kt0, kt1, mb, nb;
            split_item(sf_it, num_tiles, splits, KT, SPLIT_UNIT, tile, split, kt0, kt1);
            tile_coords(tile, tiles_m, tiles_n, mb, nb);
            const int x = 4 * kt0 + static_cast<int>(SF_ROW) * sf_g;   // 4 scale bytes per k-tile
            const uint32_t stg = sb + G::OFF_STG;
            // debug build: the boxes' innermost coordinate is a multiple of 16 bytes
            if (QG_IN_BOUNDS(err, x % 16 == 0)) {
                mbar_arrive_expect_tx(sf_full, (BM + BN) * SF_ROW);   // the two boxes' bytes
                tma_load_2d(stg, &tmSA, sf_full, x, mb * BM);
                tma_load_2d(stg + G::STG_A, &tmSB, sf_full, x, nb * BN);
            } else {
                mbar_arrive(sf_full);
            }
            ++sf_issued;
            if (++sf_g == (kt1 - kt0 + SF_GROUP - 1) / SF_GROUP) {
                sf_g = 0;
                sf_it += static_cast<int>(gridDim.x);
            }
        };
        const uint64_t keep_policy = l2_policy_evict_last();
        // current scale group in registers: [half of the group][line lane + 32 c (+ 128 h)]
        uint4 ra[2][4], rb[2][G::SFB_GROUPS][4];
        uint32_t stage = 0, phase = 0;
        for (int it = blockIdx.x; it < num_items && ok; it += gridDim.x) {
            int tile, split, kt0, kt1, mb, nb;
            split_item(it, num_tiles, splits, KT, SPLIT_UNIT, tile, split, kt0, kt1);
            tile_coords(tile, tiles_m, tiles_n, mb, nb);
            const int m0 = mb * BM, n0 = nb * BN;
            for (int kt = kt0; kt < kt1; ++kt) {
                if constexpr (SFM == SFM_TMA) {
                    if ((kt - kt0) % SF_GROUP == 0) {
                        const int q = sf_seq++;
                        if (q == 0 && lane == 0) issue_sf();
                        if (!mbar_wait(sf_full, q & 1, timeout_ns)) {
                            ok = false;
                            break;
                        }
                        sf_waited = q + 1;
                        const uint32_t stg = sb + G::OFF_STG;
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                ra[hf][c] = ld_shared_v4(stg + (lane + 32 * c) * SF_ROW + 16 * hf);
#pragma unroll
                            for (int h = 0; h < G::SFB_GROUPS; ++h)
#pragma unroll
                                for (int c = 0; c < 4; ++c)
                                    rb[hf][h][c] = ld_shared_v4(stg + G::STG_A +
                                                                (lane + 32 * c + 128 * h) * SF_ROW + 16 * hf);
                        }
                        // the whole group is in registers: refill the slot with the next one
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) issue_sf();
                    }
                }
                if (!mbar_wait(empty_bar(stage), phase ^ 1, timeout_ns)) {
                    ok = false;
                    break;
                }
                // debug build: the copies' innermost coordinates are multiples of 16 bytes
                if (!QG_IN_BOUNDS(err, (kt * BK) % 16 == 0)) {
                    ok = false;
                    break;
                }
                const uint32_t sA = sb + G::OFF_A + stage * G::A_BYTES;
                const uint32_t sB = sb + G::OFF_B + stage * G::B_BYTES;
                if (lane == 0) {
                    mbar_arrive_expect_tx(full_bar(stage), G::A_BYTES + G::B_BYTES);
                    tma_load_2d(sA, &tmA, full_bar(stage), kt * BK, m0);
                    // B panels are re-read by every row-block group: keep them in L2
                    tma_load_2d_hint(sB, &tmB, full_bar(stage), kt * BK, n0, keep_policy);
                }
                // Scale bytes: row r's 4 bytes for this k-tile go to word (r / 32) of 16-byte
                // line (r % 32) of its 128-row group.
                const int kb0 = kt * 4;
                const uint32_t nbytes = static_cast<uint32_t>(min(4, nkb - kb0));
                const uint32_t sSFA = sb + G::OFF_SFA + stage * G::SFA_BYTES;
                const uint32_t sSFB = sb + G::OFF_SFB + stage * G::SFB_BYTES;
                if constexpr (SFM == SFM_TMA) {
                    const int j = kt % 4;                          // kt0 % 4 == 0
                    const bool hi = ((kt - kt0) % SF_GROUP) >= 4;
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        if ((hf == 1) != hi) continue;
                        st_shared_v4(sSFA + lane * 16, word_of(ra[hf][0], j), word_of(ra[hf][1], j),
                                     word_of(ra[hf][2], j), word_of(ra[hf][3], j));
#pragma unroll
                        for (int h = 0; h < G::SFB_GROUPS; ++h)
                            st_shared_v4(sSFB + h * 512 + lane * 16, word_of(rb[hf][h][0], j),
                                         word_of(rb[hf][h][1], j), word_of(rb[hf][h][2], j),
                                         word_of(rb[hf][h][3], j));
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(full_bar(stage));
                } else if constexpr (SFM == SFM_CPASYNC) {
                    // 4-byte aligned scale rows: asynchronous copies, arrival when they land
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int r = m0 + 32 * c + static_cast<int>(lane);
                        const bool v = r < M;
                        const uint8_t *src = v ? sfa + static_cast<int64_t>(r) * lds_a + kb0 : sfa;
                        cp_async_4(sSFA + lane * 16 + c * 4, src, v ? nbytes : 0u);
                    }
#pragma unroll
                    for (int h = 0; h < G::SFB_GROUPS; ++h) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const int r = n0 + 128 * h + 32 * c + static_cast<int>(lane);
                            const bool v = r < N;
                            const uint8_t *src = v ? sfb + static_cast<int64_t>(r) * lds_b + kb0 : sfb;
                            cp_async_4(sSFB + h * 512 + lane * 16 + c * 4, src, v ? nbytes : 0u);
                        }
                    }
                    cp_async_arrive_noinc(full_bar(stage));
                } else {
                    // any scale stride: byte loads, then a proxy fence before the arrival
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int r = m0 + 32 * c + static_cast<int>(lane);
                        const uint32_t w =
                            r < M ? load_scale_word(sfa + static_cast<int64_t>(r) * lds_a + kb0, nbytes) : 0u;
                        st_shared_u32(sSFA + lane * 16 + c * 4, w);
                    }
#pragma unroll
                    for (int h = 0; h < G::SFB_GROUPS; ++h) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const int r = n0 + 128 * h + 32 * c + static_cast<int>(lane);
                            const uint32_t w =
                                r < N ? load_scale_word(sfb + static_cast<int64_t>(r) * lds_b + kb0, nbytes) : 0u;
                            st_shared_u32(sSFB + h * 512 + lane * 16 + c * 4, w);
                        }
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(full_bar(stage));
                }
                ++issued;
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        if (!ok && lane == 0) atomicOr(err, ERR_PRODUCER);
        // Drain: every load this warp issued has landed before the CTA may exit.
        for (int i = max(0, issued - S); i < issued; ++i) {
            if (!mbar_wait(full_bar(i % S), (i / S) & 1, timeout_ns)) {
                if (lane == 0) atomicOr(err, ERR_DRAIN);
                break;
            }
        }
        if constexpr (SFM == SFM_TMA) {
            // groups requested but never waited for (at most the one prefetched ahead)
            const int last = __shfl_sync(0xffffffffu, sf_issued, 0);
            for (int q = sf_waited; q < last; ++q)
                if (!mbar_wait(sf_full, q & 1, timeout_ns)) {
                    if (lane == 0) atomicOr(err, ERR_DRAIN);
                    break;
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA issuer
        // The whole warp runs the loop and its waits, one elected lane issues; descriptors of
        // stage 0 computed once, stage s adding s * bytes / 16 to the start-address field.
        const uint64_t adesc0 = smem_desc(sb + G::OFF_A, 16, 1024, SWZ_128B);
        const uint64_t bdesc0 = smem_desc(sb + G::OFF_B, 16, 1024, SWZ_128B);
        const uint64_t sfa0 = smem_desc(sb + G::OFF_SFA, 0, 128, SWZ_NONE);
        const uint64_t sfb0 = smem_desc(sb + G::OFF_SFB, 0, 128, SWZ_NONE);
        uint32_t stage = 0, phase = 0, acc_it = 0;
        bool ok = true;
        const uint32_t idesc = mx_idesc(BN);
        for (int it = blockIdx.x; it < num_items && ok; it += gridDim.x) {
            int tile, split, kt0, kt1;
            split_item(it, num_tiles, splits, KT, SPLIT_UNIT, tile, split, kt0, kt1);
            const uint32_t ab = acc_it % G::ACC_BUFS;   // accumulator buffer of this item
            if (!mbar_wait_warp(tmem_empty(ab), ((acc_it / G::ACC_BUFS) & 1) ^ 1, timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            for (int kt = kt0; kt < kt1; ++kt) {
                if (!mbar_wait_warp(full_bar(stage), phase, timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sf_col = tmem_base + G::SF_COL0 + stage * SF_COLS_PER_STAGE;
                const uint64_t sfa = sfa0 + stage * (G::SFA_BYTES >> 4);
                const uint64_t sfb = sfb0 + stage * (G::SFB_BYTES >> 4);
                const uint64_t adesc = adesc0 + stage * (G::A_BYTES >> 4);
                const uint64_t bdesc = bdesc0 + stage * (G::B_BYTES >> 4);
                if (elect_one()) {
                    if constexpr (SFM == SFM_CPASYNC)
                        fence_proxy_async_smem();  // cp.async (generic proxy) -> tcgen05.cp reads
                    tc_cp_32x128b_warpx4(sf_col, sfa);
#pragma unroll
                    for (int h = 0; h < G::SFB_GROUPS; ++h)
                        tc_cp_32x128b_warpx4(sf_col + 4 + 4 * h, sfb + h * (512 >> 4));
#pragma unroll
                    for (uint32_t j = 0; j < BK / 32; ++j) {
                        // advance 32 bytes of K inside the 128-byte swizzle row
                        mma_mxf8(tmem_base + ab * BN, adesc + 2 * j, bdesc + 2 * j,
                                 idesc | (j << 4) | (j << 29), sf_col, sf_col + 4,
                                 (kt > kt0 || j > 0) ? 1u : 0u);
                    }
                    tc_commit(empty_bar(stage));
                }
                __syncwarp();
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) break;
            if (elect_one()) tc_commit(tmem_full(ab));
            __syncwarp();
            ++acc_it;
        }
        // Drain: all MMAs and TMEM copies of this CTA have completed before TMEM is freed (the
        // commit comes from the lane that issued them: elect.sync picks the lowest active lane).
        if (elect_one()) {
            if (!ok) atomicOr(err, ERR_MMA);
            tc_commit(drain_bar);
        }
        __syncwarp();
        if (!mbar_wait(drain_bar, 0, timeout_ns) && lane == 0) atomicOr(err, ERR_DRAIN);
    } else {
        // ---------------------------------------------------------------- epilogue
        const uint32_t q = warp & 3;  // TMEM lane quarter this warp may read
        uint32_t acc_it = 0;
        for (int it = blockIdx.x; it < num_items; it += gridDim.x) {
            int tile, split, kt0, kt1, mb, nb;
            split_item(it, num_tiles, splits, KT, SPLIT_UNIT, tile, split, kt0, kt1);
            tile_coords(tile, tiles_m, tiles_n, mb, nb);
            const uint32_t ab = acc_it % G::ACC_BUFS;
            if (!mbar_wait_sleep(tmem_full(ab), (acc_it / G::ACC_BUFS) & 1, timeout_ns, 128)) {
                if (lane == 0) atomicOr(err, ERR_EPILOGUE);
                break;
            }
            tc_fence_after();
            if (splits > 1)    // this k range's unrounded sum into its partial plane
                partial_tile<BN>(tmem_base + ab * BN, q, lane, P + split * plane, ldp, mb * BM,
                                 nb * BN, M, tmem_empty(ab), sb + G::OFF_EPI + (warp - 2) * 2048);
            else
                epilogue_tile<BN>(tmem_base + ab * BN, q, lane, C, ldc, mb * BM, nb * BN, M, N,
                                  c_vec != 0, tmem_empty(ab), sb + G::OFF_EPI + (warp - 2) * 2048,
                                  epi);
            ++acc_it;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

template <int BN, int SFM>
cudaError_t launch_bn(const qgemm_tensor *A, const qgemm_tensor *B, __half *C, int64_t ldc,
                      int splits, float *P, int64_t ldp, const qgi::LaunchCtx &ctx,
                      bool *encode_ok) {
    using G = Cfg<BN>;
    const int M = static_cast<int>(A->rows), N = static_cast<int>(B->rows),
              K = static_cast<int>(A->k);
    CUtensorMap tmA, tmB, tmSA, tmSB;
    *encode_ok = qgi::encode_tma_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A->data, K, M, A->ld, BK,
                                    BM, CU_TENSOR_MAP_SWIZZLE_128B) &&
                 qgi::encode_tma_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B->data, K, N, B->ld, BK,
                                    BN, CU_TENSOR_MAP_SWIZZLE_128B);
    if (*encode_ok && SFM == SFM_TMA)
        *encode_ok = qgi::encode_tma_2d(&tmSA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A->scales, K / 32, M,
                                        A->lds, SF_ROW, BM, CU_TENSOR_MAP_SWIZZLE_NONE) &&
                     qgi::encode_tma_2d(&tmSB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B->scales, K / 32, N,
                                        B->lds, SF_ROW, BN, CU_TENSOR_MAP_SWIZZLE_NONE);
    else
        tmSA = tmA, tmSB = tmB;   // unused by the other scale routes
    if (!*encode_ok) return cudaErrorInvalidValue;
    auto kern = mxfp8_gemm_kernel<BN, SFM>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int64_t items = static_cast<int64_t>((M + BM - 1) / BM) * ((N + BN - 1) / BN) * splits;
    const int grid = items < ctx.num_sms ? static_cast<int>(items) : ctx.num_sms;
    const int c_vec = (reinterpret_cast<uintptr_t>(C) % 16 == 0 && ldc % 8 == 0) ? 1 : 0;
    kern<<<grid, THREADS, G::SMEM_BYTES, ctx.stream>>>(tmA, tmB, tmSA, tmSB, A->scales, A->lds,
                                                        B->scales, B->lds, C, ldc, c_vec, M, N, K,
                                                        splits, P, ldp, ctx.epi, ctx.err,
                                                        ctx.timeout_ns);
    return cudaGetLastError();
}

template <int BN>
cudaError_t launch_sfm(const qgemm_tensor *A, const qgemm_tensor *B, __half *C, int64_t ldc,
                       int splits, float *P, int64_t ldp, const qgi::LaunchCtx &ctx,
                       bool *encode_ok) {
    auto al = [](const qgemm_tensor *t, int a) {
        return reinterpret_cast<uintptr_t>(t->scales) % a == 0 && t->lds % a == 0;
    };
    if (al(A, 16) && al(B, 16))
        return launch_bn<BN, SFM_TMA>(A, B, C, ldc, splits, P, ldp, ctx, encode_ok);
    if (al(A, 4) && al(B, 4))
        return launch_bn<BN, SFM_CPASYNC>(A, B, C, ldc, splits, P, ldp, ctx, encode_ok);
    return launch_bn<BN, SFM_BYTES>(A, B, C, ldc, splits, P, ldp, ctx, encode_ok);
}

// Split-K on the one-CTA route: when the output has at most half as many tiles as the GPU has
// SMs, each tile's k-tiles are shared out over up to SMs / tiles CTAs (whole units of four
// k-tiles each), which write fp32 partial planes that splitk_reduce.cu adds in split order.
// Partial planes are M rows of ldp = tiles_n * BN floats.
struct SplitPlan {
    int bn, splits;
    int64_t ldp;
    size_t bytes;
};

SplitPlan split_plan(const qgemm_tensor *A, const qgemm_tensor *B, int num_sms, bool allow) {
    const int64_t M = A->rows, N = B->rows, K = A->k;
    SplitPlan p;
    p.bn = N > 128 ? 256 : 128;
    const int64_t tiles_n = (N + p.bn - 1) / p.bn;
    const int64_t tiles = ((M + BM - 1) / BM) * tiles_n;
    const int64_t units = ((K + BK - 1) / BK + SPLIT_UNIT - 1) / SPLIT_UNIT;
    int64_t s = 1;
    if (allow && 2 * tiles <= num_sms) s = std::min<int64_t>(num_sms / tiles, units);
    p.splits = static_cast<int>(s < 1 ? 1 : s);
    p.ldp = tiles_n * p.bn;
    p.bytes = p.splits > 1 ? static_cast<size_t>(p.splits) * M * p.ldp * sizeof(float) : 0;
    return p;
}

}  // namespace

namespace qgi {

size_t mxfp8_scratch_bytes(const qgemm_tensor *A, const qgemm_tensor *B, int num_sms) {
    if (A->rows == 0 || B->rows == 0 || A->k == 0) return 0;
    if (mxfp8_pair_eligible(A, B)) return mxfp8_pair_scratch_bytes(A, B);
    return split_plan(A, B, num_sms, true).bytes;
}

cudaError_t launch_mxfp8(const qgemm_tensor *A, const qgemm_tensor *B, __half *C, int64_t ldc,
                         const LaunchCtx &ctx, bool *encode_ok, bool allow_split) {
    // CTA pairs (mxfp8_pair.cu, scales repacked into pooled scratch) when both operands span
    // more than one 128-row block; otherwise one CTA per tile.  BN = 256 with one accumulator
    // measured faster than BN = 224 with two at 8192^3.
    if (mxfp8_pair_eligible(A, B)) {
        void *scratch = nullptr;
        cudaError_t e = scratch_alloc(mxfp8_pair_scratch_bytes(A, B), ctx, &scratch);
        if (e != cudaSuccess) return e;
        e = launch_mxfp8_pair(A, B, C, ldc, scratch, ctx, encode_ok);
        const cudaError_t f = scratch_free(scratch, ctx);
        return e != cudaSuccess ? e : f;
    }
    const SplitPlan p = split_plan(A, B, ctx.num_sms, allow_split);
    void *ws = nullptr;
    if (p.splits > 1) {
        cudaError_t e = scratch_alloc(p.bytes, ctx, &ws);
        if (e != cudaSuccess) return e;
    }
    float *P = static_cast<float *>(ws);
    cudaError_t e = p.bn == 256 ? launch_sfm<256>(A, B, C, ldc, p.splits, P, p.ldp, ctx, encode_ok)
                                : launch_sfm<128>(A, B, C, ldc, p.splits, P, p.ldp, ctx, encode_ok);
    if (e == cudaSuccess && p.splits > 1)
        e = launch_splitk_reduce(P, p.splits, p.ldp, static_cast<int>(A->rows),
                                 static_cast<int>(B->rows), C, ldc, ctx);
    const cudaError_t f = scratch_free(ws, ctx);
    return e != cudaSuccess ? e : f;
}

}  // namespace qgi
