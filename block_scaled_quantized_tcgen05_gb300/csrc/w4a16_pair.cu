// w4a16_pair.cu -- weight-only int4 GEMM on CTA pairs with the dequantised weights in TMEM.
//
// C[M, N] = fp16_rn( sum_k A[m, k] * q(W[n, k]) * 2^(SW[n, k/32] - 127) ),  fp32 accumulation.
//
// "TensorOps: quantized matmul ..." (sections "Revised kernel strategy" and "M2 = block-32 fp16
// scaling") dequantises each 32-block of int4 weights into on-chip memory and runs the half x
// half product there; its escape-hatch note asks for the dequantised weights to go straight into
// the operand the matrix unit reads.  On GB300 the tensor core can read its A operand from TMEM,
// so this kernel computes the transposed product D[n, m] = sum_k W[n, k] A[m, k] with the weights
// as the A operand in TMEM and the activations as the B operand in shared memory:
//
//   * a cluster of two CTAs computes a 256 (weight rows) x 256 (tokens) tile with
//     tcgen05.mma.cta_group::2.kind::f16; each CTA holds 128 weight rows in its TMEM and 128
//     token rows of A in its shared memory;
//   * converter warps -- two per TMEM lane quarter, taking alternate k-tiles -- read the packed
//     int4 bytes of their 32 weight rows (one row per lane, landed by TMA), turn each 32-block
//     into fp16 with its scale in registers and write the 64-element k-tile into the stage's TMEM
//     slot with one tcgen05.st (32 columns, two fp16 per column, even k in the low half);
//   * the dequantised weights never touch shared memory, whose bandwidth (TMA writes plus tensor
//     reads) is what bounds a weight-in-shared-memory design;
//   * the epilogue reads D (lane = weight row n, column = token m); each lane owns one output
//     column, so it writes its 32 tokens of a chunk as 2-byte stores into the warp's shared
//     staging, laid out [token][32 columns] (one 64-byte row per store instruction, no bank
//     conflicts); the accumulator is released right after the last TMEM read and the staged
//     32 x 32 blocks go out as TMA tensor stores, so no tile waits for the output traffic (all pairs
//     reach their epilogue together and the stores come in bursts).  C not 16-byte aligned, or
//     its row stride not a multiple of 8, takes direct 2-byte global stores instead.
//
// Hand-off as in mxfp8_pair.cu: the leader issues every MMA from one thread and waits once per
// stage on its full barrier, which collects both CTAs' activation bytes and one relaxed arrival
// from each converter warp of both CTAs after its tcgen05.st completed; commits are multicast;
// every wait is bounded.  Used for K % 512 == 0 with 16-byte aligned scale rows (scales are read
// 16 bytes = 8 k-tiles at a time); other shapes take w4a16_gemm.cu.  With few tiles (a few tokens
// against many weight rows) and no accumulation, the SPLIT instance cuts each tile's K into whole
// 512-wide slices over several pairs, which write fp32 partial planes for splitk_reduce.cu.  Scale bytes outside the
// fold window convert to zero weights (w4a16_convert.cuh); when the output is accumulated, the
// columns of outlier rows are left to w4a16_outlier.cu, which runs next and needs the old C.
//
// The same kernel, instantiated with SB = 2, runs the custom-format escape hatch: int4 weights
// with arbitrary fp16 scales per 32-block ("TensorOps: quantized matmul ...", "M2 = block-32 fp16
// scaling": each weight dequantised into half as q times its block's half scale).  The
// converters then multiply the exact fp16 q by the fp16 scale with one rounding (mul.rn.f16x2),
// which is that recipe's half multiply; scales are read 16 bytes = 4 k-tiles at a time, so that
// instance needs K % 256 == 0 and 16-byte aligned scale rows, and takes every M and N.
#include "qgemm_common.cuh"
#include "qgemm_debug.cuh"
#include "qgemm_internal.h"
#include "qgemm_ptx.cuh"
#include "w4a16_convert.cuh"

#include <algorithm>

namespace {

using namespace qg;

constexpr int BW = 128;                 // weight rows per CTA (256 per pair: the MMA's M)
constexpr int BT = 256;                 // tokens per pair tile (the MMA's N), 128 per CTA
constexpr int BK = 64;                  // k per stage
constexpr int STAGES = 8;
constexpr int EPI_WARPS = 8;            // two per lane quarter, one per half of the 256 tokens
constexpr int CONV_WARP0 = 2 + EPI_WARPS;
constexpr int CONV_WARPS = 8;           // two per lane quarter, alternate k-tiles
constexpr int THREADS = 32 * (CONV_WARP0 + CONV_WARPS);
constexpr int SPLIT_UNIT = 8;           // split-K ranges: whole 512-wide slices of K (8 k-tiles)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t A_COL0 = 256;        // weight slots after the 256-column accumulator
constexpr uint32_t A_COLS = BK / 2;     // 32 columns per stage

constexpr uint32_t X_BYTES = (BT / 2) * BK * 2;   // 16 KB: this CTA's 128 token rows
constexpr uint32_t RAW_BYTES = BW * (BK / 2);     // 4 KB: packed int4 of this CTA's weight rows
constexpr uint32_t STAGE_TX = 2 * X_BYTES;        // both CTAs' activations, on the leader
constexpr uint32_t OFF_X = 0;
constexpr uint32_t OFF_RAW = OFF_X + STAGES * X_BYTES;
constexpr uint32_t EPI_BYTES = 4 * 32 * 32 * 2;     // per epilogue warp: 4 chunks of 32 x 32 fp16
constexpr uint32_t OFF_EPI = OFF_RAW + STAGES * RAW_BYTES;
constexpr uint32_t OFF_BAR = OFF_EPI + EPI_WARPS * EPI_BYTES;
// full[S] (leader), empty[S], raw_full[S], tmem_full, tmem_empty (leader), drain, then the slot
constexpr uint32_t OFF_SLOT = OFF_BAR + (3 * STAGES + 3) * 8;
constexpr uint32_t SMEM_BYTES = OFF_SLOT + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(A_COL0 + STAGES * A_COLS <= TMEM_COLS, "TMEM budget");

// kind::f16: D fp32, A and B fp16, K-major, N = 256 tokens, M = 256 weight rows (pair).
constexpr uint32_t IDESC = (1u << 4) | (static_cast<uint32_t>(BT >> 3) << 17) |
                           (static_cast<uint32_t>(256 >> 4) << 24);

__device__ __forceinline__ uint4 ld_nc_v4(const uint8_t *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

__device__ __forceinline__ void st_global_cs_u16(__half *p, uint16_t v) {
    asm volatile("st.global.cs.b16 [%0], %1;" ::"l"(p), "h"(v) : "memory");
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// SB: bytes per block scale (1: UE8M0 byte, 2: fp16).  lds is in bytes.
template <int SB, bool SPLIT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
w4a16_pair_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                  const __grid_constant__ CUtensorMap tmC, int c_tma,
                  const uint8_t *__restrict__ scales, int64_t lds,
                  const uint8_t *__restrict__ wdata, int64_t ldw, __half *__restrict__ C,
                  int64_t ldc, int M, int N, int K, int splits, float *__restrict__ P,
                  int64_t ldp, int epi, unsigned *err, uint64_t timeout_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_1024(smem_raw);
    // the split-K reduction or the outlier-row pass may take the room this CTA leaves
    griddep_launch_dependents();
    const uint32_t sb = smem_u32(smem);
    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();      // 0 = leader
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;

    auto full_bar = [&](int s) { return sb + OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sb + OFF_BAR + 8u * (STAGES + s); };
    auto raw_full = [&](int s) { return sb + OFF_BAR + 8u * (2 * STAGES + s); };
    const uint32_t tmem_full = sb + OFF_BAR + 8u * (3 * STAGES);
    const uint32_t tmem_empty = tmem_full + 8;
    const uint32_t drain_bar = tmem_full + 16;
    volatile uint32_t *slot = reinterpret_cast<volatile uint32_t *>(smem + OFF_SLOT);

    // tiles: weight-row blocks of 256 (the "m" of tile_coords) x token blocks of 256
    const int tiles_w = (N + 2 * BW - 1) / (2 * BW);
    const int tiles_t = (M + BT - 1) / BT;
    const int num_tiles = tiles_w * tiles_t;
    const int KT = K / BK;
    // work items (tile, k range): with splits > 1 each tile's K is cut into `splits` ranges of
    // whole scale groups (SPLIT_UNIT k-tiles), each summed into its own fp32 partial plane
    const int num_items = num_tiles * splits;
    const int64_t plane = static_cast<int64_t>(M) * ldp;
    // (the instance without a split compiles to whole tiles over all of K)
    auto item_of = [&](int it, int &tile, int &split, int &kt0, int &kt1) {
        if constexpr (SPLIT) {
            split_item(it, num_tiles, splits, KT, SPLIT_UNIT, tile, split, kt0, kt1);
        } else {
            tile = it;
            split = 0;
            kt0 = 0;
            kt1 = KT;
        }
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1 + 2 * (CONV_WARPS / 2));   // expect_tx + converters of a stage
            mbar_init(empty_bar(s), 1);                          // leader's multicast commit
            mbar_init(raw_full(s), 1);                           // this CTA's packed-int4 TMA
        }
        mbar_init(tmem_full, 1);
        mbar_init(tmem_empty, 2 * EPI_WARPS);   // one lane of each epilogue warp of both CTAs
        mbar_init(drain_bar, 1);
        fence_barrier_init();
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
        if (c_tma) tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(const_cast<uint32_t *>(slot)), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();                   // barriers of both CTAs initialised before remote use
    tc_fence_after();
    const uint32_t tmem_base = *slot;

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        // The whole warp runs the loop and waits; one elected lane issues the copies.
        {
            uint32_t stage = 0, phase = 0;
            int issued = 0;
            bool ok = true;
            for (int it = pair; it < num_items && ok; it += npairs) {
                int tile, split, kt0, kt1, wb, tb;
                item_of(it, tile, split, kt0, kt1);
                tile_coords(tile, tiles_w, tiles_t, wb, tb);
                const int w0 = wb * 2 * BW + static_cast<int>(rank) * BW;     // this CTA's weights
                const int t0 = tb * BT + static_cast<int>(rank) * (BT / 2);   // this CTA's tokens
                for (int kt = kt0; kt < kt1; ++kt) {
                    if (!mbar_wait_warp(empty_bar(stage), phase ^ 1, timeout_ns)) {
                        ok = false;
                        break;
                    }
                    // debug build: the copies' innermost coordinates are multiples of 16 bytes
                    if (!QG_IN_BOUNDS(err, (kt * BK) % 8 == 0 && (kt * (BK / 2)) % 16 == 0)) {
                        ok = false;
                        break;
                    }
                    const uint32_t lead_full = map_to_cta(full_bar(stage), 0);
                    if (elect_one()) {
                        if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), STAGE_TX);
                        tma_load_2d_pair(sb + OFF_X + stage * X_BYTES, &tmX, lead_full, kt * BK,
                                         t0);
                        mbar_arrive_expect_tx(raw_full(stage), RAW_BYTES);
                        tma_load_2d(sb + OFF_RAW + stage * RAW_BYTES, &tmW, raw_full(stage),
                                    kt * (BK / 2), w0);
                    }
                    __syncwarp();
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok && lane == 0) atomicOr(err, ERR_PRODUCER);
            for (int i = max(0, issued - STAGES); i < issued; ++i) {
                const bool drained =
                    mbar_wait(raw_full(i % STAGES), (i / STAGES) & 1, timeout_ns) &&
                    (rank != 0 ||
                     mbar_wait_cluster(full_bar(i % STAGES), (i / STAGES) & 1, timeout_ns));
                if (!__all_sync(0xFFFFFFFFu, drained)) {
                    if (lane == 0) atomicOr(err, ERR_DRAIN);
                    break;
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (rank == 0) {
            // --------------------------------------------------------- MMA issuer
            // The whole warp runs the loop and waits; one elected lane issues (a loop run by one
            // lane alone issues measurably slower, more so beside the converter warps' ALU work).
            const uint64_t bdesc0 = smem_desc(sb + OFF_X, 16, 1024, SWZ_128B);
            uint32_t acc_phase = 0, stage = 0, phase = 0;
            bool ok = true;
            for (int it = pair; it < num_items && ok; it += npairs) {
                int tile, split, kt0, kt1;
                item_of(it, tile, split, kt0, kt1);
                if (!__all_sync(0xFFFFFFFFu,
                                mbar_wait_cluster(tmem_empty, acc_phase ^ 1, timeout_ns))) {
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
                    const uint32_t a_col = tmem_base + A_COL0 + stage * A_COLS;
                    const uint64_t bdesc = bdesc0 + stage * (X_BYTES >> 4);
                    if (elect_one()) {
                        mma_f16_pair_ta(tmem_base, a_col, bdesc, IDESC, kt > kt0 ? 1u : 0u);
#pragma unroll
                        for (uint32_t j = 1; j < BK / 16; ++j)
                            mma_f16_pair_ta(tmem_base, a_col + 8 * j, bdesc + 2 * j, IDESC, 1u);
                        tc_commit_pair(empty_bar(stage), 3);
                    }
                    __syncwarp();
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                if (elect_one()) tc_commit_pair(tmem_full, 3);
                __syncwarp();
                acc_phase ^= 1;
            }
            if (elect_one()) {
                if (!ok) atomicOr(err, ERR_MMA);
                tc_commit_pair(drain_bar, 3);
            }
        }
        __syncwarp();
        // both CTAs: every pair MMA writing this CTA's TMEM has completed before it is freed
        if (!mbar_wait(drain_bar, 0, timeout_ns) && lane == 0) atomicOr(err, ERR_DRAIN);
    } else if (warp >= CONV_WARP0) {
        // ----------------------------------------------------------------- converters
        // Lane i of a warp of lane quarter q dequantises weight row 32 q + i of this CTA's 128;
        // the two warps of a quarter take the even and the odd stages of the sequence.
        const uint32_t q = warp & 3;
        const int parity = static_cast<int>(warp - CONV_WARP0) >> 2;
        const uint32_t lead_full = map_to_cta(full_bar(0), 0);
        const int r = static_cast<int>(q * 32 + lane);
        constexpr int SPG = 8 / SB;              // k-tiles per 16-byte scale group
        // this pair's work items in order (ti = 0, 1, ...): item pair + ti * npairs, whose
        // k-tiles [kt0, kt1) hold whole scale groups kt0 / SPG .. kt1 / SPG - 1
        auto item_range = [&](int ti, int &tile, int &kt0, int &kt1) -> bool {
            const int it = pair + ti * npairs;
            if (it >= num_items) return false;
            int split;
            item_of(it, tile, split, kt0, kt1);
            return true;
        };
        int total = 0;                           // this pair's k-tiles over all its items
        for (int ti = 0;; ++ti) {
            int tile, a0, a1;
            if (!item_range(ti, tile, a0, a1)) break;
            total += a1 - a0;
        }
        // Scale group prefetch cursor: group nxt_g of item nxt_ti, whose groups end at nxt_g1
        // and whose scale row for this lane starts at nxt_row (null past N or past the last
        // item).  The item's tile and range are looked up once per item, not per group.
        int nxt_ti = 0, nxt_g = 0, nxt_g1 = 0;
        const uint8_t *nxt_row = nullptr;
        auto load_item = [&](int ti) {
            int tile, a0, a1;
            nxt_ti = ti;
            nxt_row = nullptr;
            nxt_g = nxt_g1 = 0;
            if (!item_range(ti, tile, a0, a1)) return;
            int wb, tb;
            tile_coords(tile, tiles_w, tiles_t, wb, tb);
            const int n = wb * 2 * BW + static_cast<int>(rank) * BW + r;
            if (n < N) nxt_row = scales + static_cast<int64_t>(n) * lds;
            nxt_g = a0 / SPG;
            nxt_g1 = a1 / SPG;
        };
        // rows past N: scale 1 (their weights are TMA zero fill, so any finite scale gives 0)
        constexpr uint32_t ONE = SB == 1 ? 0x7F7F7F7Fu : 0x3C003C00u;
        const uint4 unit = make_uint4(ONE, ONE, ONE, ONE);
        auto fetch = [&]() -> uint4 {
            return nxt_row != nullptr && nxt_g < nxt_g1 ? ld_nc_v4(nxt_row + 16 * nxt_g) : unit;
        };
        auto advance = [&]() {
            if (++nxt_g >= nxt_g1) load_item(nxt_ti + 1);
        };
        load_item(0);
        int cur_ti = nxt_ti, cur_g = nxt_g;
        uint4 cur = total > 0 ? fetch() : unit;
        advance();
        uint4 nxt = total > 0 ? fetch() : unit;
        // each warp walks only its own k-tiles, every other one (an item's k-tiles are whole
        // scale groups of SPG >= 4, an even count, so both parities visit every group in order)
        uint32_t stage = static_cast<uint32_t>(parity), phase = 0;
        int ti = 0, it_kt0, it_kt1;
        {
            int tile;
            if (!item_range(0, tile, it_kt0, it_kt1)) it_kt0 = it_kt1 = 0;
        }
        int kt = it_kt0 + parity;
        for (int it = parity; it < total; it += 2) {
            const int g = kt / SPG;
            if (ti != cur_ti || g != cur_g) {    // move to the next scale group, prefetch one more
                cur = nxt;
                cur_ti = nxt_ti;
                cur_g = nxt_g;
                advance();
                nxt = fetch();
            }
            if (!mbar_wait(raw_full(stage), phase, timeout_ns)) {
                if (lane == 0) atomicOr(err, ERR_PRODUCER);
                break;
            }
            tc_fence_after();   // the MMAs that last read this TMEM slot have completed
            const uint8_t *raw = smem + OFF_RAW + stage * RAW_BYTES + r * (BK / 2);
            const uint4 lo = *reinterpret_cast<const uint4 *>(raw);        // k  0..31
            const uint4 hi = *reinterpret_cast<const uint4 *>(raw + 16);   // k 32..63
            // this stage's two block scales: bytes 2 (kt % 8), + 1 of the group (UE8M0), or
            // the fp16 pair in word kt % 4 (fp16 scales)
            const int sbyte = SB == 1 ? (kt & 7) * 2 : (kt & 3) * 4;
            const int wsel = sbyte >> 2;
            const uint32_t word = wsel == 0 ? cur.x : wsel == 1 ? cur.y : wsel == 2 ? cur.z : cur.w;
            uint32_t out[32];
            if constexpr (SB == 2) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t s2 = __byte_perm(word, 0u, h ? 0x3232u : 0x1010u);
                    const uint4 d = h ? hi : lo;
                    const uint32_t words[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        uint32_t o[4];
                        i4x8_to_f16(words[w], s2, o);   // exact q, then one rounding of q*s
#pragma unroll
                        for (int j = 0; j < 4; ++j) out[16 * h + 4 * w + j] = o[j];
                    }
                }
            } else {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t e = (word >> (8 * ((sbyte & 3) + h))) & 0xFFu;
                    const uint4 d = h ? hi : lo;
                    const uint32_t words[4] = {d.x, d.y, d.z, d.w};
                    if (fused_ok(e)) {
                        uint32_t s2, c2;
                        fused_consts(e, s2, c2);
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            uint32_t o[4];
                            i4x8_to_f16_fused(words[w], s2, c2, o);
#pragma unroll
                            for (int j = 0; j < 4; ++j) out[16 * h + 4 * w + j] = o[j];
                        }
                    } else {
                        const uint32_t s2 = ue8m0_to_f16x2(e);
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            uint32_t o[4];
                            i4x8_to_f16(words[w], s2, o);
#pragma unroll
                            for (int j = 0; j < 4; ++j) out[16 * h + 4 * w + j] = o[j];
                        }
                    }
                }
            }
            tmem_st_32x32b_x32(tmem_base + ((q * 32) << 16) + A_COL0 + stage * A_COLS, out);
            tmem_wait_st();
            tc_fence_before();
            // the raw weights were read through the generic proxy; the slot's next fill is a TMA write
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive_relaxed_cluster(lead_full + 8u * stage);
            stage += 2;
            if (stage >= STAGES) {
                stage -= STAGES;
                phase ^= 1;
            }
            if ((kt += 2) >= it_kt1) {           // on to this warp's first k-tile of the next item
                const int over = kt - it_kt1;
                ++ti;
                int tile;
                if (!item_range(ti, tile, it_kt0, it_kt1)) it_kt0 = it_kt1 = 0;
                kt = it_kt0 + over;
            }
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        // Lane i of a warp of lane quarter q holds output column n = weight row 32 q + i; the
        // warp covers 128 of the tile's 256 tokens, 32 per TMEM read.
        const uint32_t q = warp & 3;
        const uint32_t half = (warp - 2) >> 2;
        const uint32_t lead_empty = map_to_cta(tmem_empty, 0);
        uint32_t acc_phase = 0;
        for (int it = pair; it < num_items; it += npairs) {
            int tile, split, kt0, kt1, wb, tb;
            item_of(it, tile, split, kt0, kt1);
            tile_coords(tile, tiles_w, tiles_t, wb, tb);
            const int n0 = wb * 2 * BW + static_cast<int>(rank) * BW + static_cast<int>(q * 32);
            const int n = n0 + static_cast<int>(lane);
            // Accumulating: an outlier row's column is left to w4a16_outlier_kernel, which needs
            // the old C (checked while the tile's MMAs run).
            bool skip = false;
            if constexpr (SB == 1) {
                if ((epi & EPI_ACC_BIT) && n < N)
                    skip = w4_row_is_outlier(scales + static_cast<int64_t>(n) * lds,
                                             wdata + static_cast<int64_t>(n) * ldw, K / 32);
            }
            if (!mbar_wait_sleep(tmem_full, acc_phase, timeout_ns, 128)) {
                if (lane == 0) atomicOr(err, ERR_EPILOGUE);
                break;
            }
            tc_fence_after();
            const int m0 = tb * BT + static_cast<int>(half) * (BT / 2);
            if constexpr (SPLIT) {
                // this k range's unrounded sums into its partial plane, [token][weight row]:
                // lane = weight row, so each store writes 32 consecutive floats of a token row
                float *pl = P + split * plane;
#pragma unroll 1
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tmem_base + ((q * 32) << 16) + half * (BT / 2) + ch * 32, v);
                    tmem_wait_ld();
                    if (ch == 3) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_relaxed_cluster(lead_empty);
                    }
                    if (n < N) {
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            const int m = m0 + ch * 32 + c;
                            if (m < M) pl[static_cast<int64_t>(m) * ldp + n] = __uint_as_float(v[c]);
                        }
                    }
                }
                acc_phase ^= 1;
                continue;
            }
            const uint32_t stg = sb + OFF_EPI + (warp - 2) * EPI_BYTES;
            if (c_tma) {   // the previous tile's stores have finished reading the staging
                if (lane == 0) bulk_wait_read<0>();
                __syncwarp();
            }
            if (c_tma && !(epi & EPI_ACC_BIT)) {
                // the whole 32 x 128 slice into registers as fp16 pairs, the accumulator handed
                // back, and only then the staging stores (the next tile's MMAs need not wait for
                // them): 2 % at 4096 x 14336 x 4096 with UE8M0 scales, about 1 % with fp16 scales
                uint32_t pk[4][16];
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tmem_base + ((q * 32) << 16) + half * (BT / 2) + ch * 32, v);
                    tmem_wait_ld();
                    if (epi & EPI_RELU_BIT) {
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            v[c] = __float_as_uint(fmaxf(__uint_as_float(v[c]), 0.0f));
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[ch][i] = pack_f16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_relaxed_cluster(lead_empty);
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        // row c of the chunk: tokens m0 + 32 ch + c, columns n0 .. n0 + 31
                        st_shared_u16(stg + ch * 2048 + (2 * i) * 64 + lane * 2,
                                      static_cast<uint16_t>(pk[ch][i] & 0xFFFFu));
                        st_shared_u16(stg + ch * 2048 + (2 * i + 1) * 64 + lane * 2,
                                      static_cast<uint16_t>(pk[ch][i] >> 16));
                    }
            } else
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem_base + ((q * 32) << 16) + half * (BT / 2) + ch * 32, v);
                tmem_wait_ld();
                if (ch == 3) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_relaxed_cluster(lead_empty);
                }
                if ((epi & EPI_RELU_BIT) && !(epi & EPI_ACC_BIT)) {   // (after the add otherwise)
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        v[c] = __float_as_uint(fmaxf(__uint_as_float(v[c]), 0.0f));
                }
                if (c_tma) {
                    // row c of the chunk: tokens m0 + 32 ch + c, columns n0 .. n0 + 31
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        st_shared_u16(stg + ch * 2048 + c * 64 + lane * 2,
                                      __half_as_ushort(__float2half_rn(__uint_as_float(v[c]))));
                } else if (n < N && !skip) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const int m = m0 + ch * 32 + c;
                        if (m < M) {
                            __half *dst = C + static_cast<int64_t>(m) * ldc + n;
                            float x = __uint_as_float(v[c]);
                            if (epi & EPI_ACC_BIT) {   // C = relu?(acc + C_old), one rounding
                                x += __half2float(*dst);
                                if (epi & EPI_RELU_BIT) x = fmaxf(x, 0.0f);
                            }
                            st_global_cs_u16(dst, __half_as_ushort(__float2half_rn(x)));
                        }
                    }
                }
            }
            if (c_tma) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch)   // blocks wholly past M or N are not stored
                        if (n0 < N && m0 + ch * 32 < M)
                            tma_store_2d(&tmC, stg + ch * 2048, n0, m0 + ch * 32);
                    bulk_commit();
                }
            }
            acc_phase ^= 1;
        }
        if (c_tma && lane == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();                   // no remote arrival or multicast targets an exited CTA
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

template <int SB>
cudaError_t launch_pair_impl(const __half *A, int64_t lda, int M, const qgemm_tensor *W,
                             __half *C, int64_t ldc, const qgi::LaunchCtx &ctx, bool *encode_ok) {
    const int N = static_cast<int>(W->rows), K = static_cast<int>(W->k);
    CUtensorMap tmX, tmW, tmC;
    *encode_ok = qgi::encode_tma_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, K, M, lda * 2, BK,
                               BT / 2, CU_TENSOR_MAP_SWIZZLE_128B) &&
                 qgi::encode_tma_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, W->data, K / 2, N, W->ld,
                               BK / 2, BW, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!*encode_ok) return cudaErrorInvalidValue;
    // output through TMA stores when C and its row stride allow a tensor map
    // (the accumulate epilogue reads the old C element by element: direct stores)
    const int c_tma = (reinterpret_cast<uintptr_t>(C) % 16 == 0 && ldc % 8 == 0 &&
                       !(ctx.epi & qgi::EPI_ACCUMULATE)) ? 1 : 0;
    if (c_tma) {
        *encode_ok = qgi::encode_tma_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, C, N, M, ldc * 2, 32, 32,
                                   CU_TENSOR_MAP_SWIZZLE_NONE);
        if (!*encode_ok) return cudaErrorInvalidValue;
    } else {
        tmC = tmX;   // unused
    }
    cudaError_t e;
    const int tiles_w = (N + 2 * BW - 1) / (2 * BW);
    const int tiles = tiles_w * ((M + BT - 1) / BT);
    // A few tokens against many weight rows leave most pairs idle: when the tiles fill at most
    // half of the pairs, each tile's K is split over up to pairs / tiles pairs (whole 512-wide
    // slices), their fp32 partial planes added in order by splitk_reduce.cu.  Not when the
    // output is accumulated: the outlier-row pass then needs the old C of its columns, which
    // the reduction would overwrite.
    const int avail = ctx.num_sms / 2;
    int splits = 1;
    if (!(ctx.epi & qgi::EPI_ACCUMULATE) && 2 * tiles <= avail)
        splits = std::min(avail / tiles, (K / BK) / SPLIT_UNIT);
    if (splits < 1) splits = 1;
    const int64_t ldp = static_cast<int64_t>(tiles_w) * 2 * BW;
    void *ws = nullptr;
    if (splits > 1) {
        e = qgi::scratch_alloc(static_cast<size_t>(splits) * static_cast<size_t>(M) *
                                   static_cast<size_t>(ldp) * sizeof(float),
                               ctx, &ws);
        if (e != cudaSuccess) return e;
    }
    float *P = static_cast<float *>(ws);
    const int items = tiles * splits;
    int pairs = avail;
    if (pairs > items) pairs = items;
    auto kern = splits > 1 ? w4a16_pair_kernel<SB, true> : w4a16_pair_kernel<SB, false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e == cudaSuccess) {
        kern<<<2 * pairs, THREADS, SMEM_BYTES, ctx.stream>>>(
            tmX, tmW, tmC, c_tma, W->scales, W->lds, W->data, W->ld, C, ldc, M, N, K, splits, P, ldp,
            ctx.epi, ctx.err, ctx.timeout_ns);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess && splits > 1) e = qgi::launch_splitk_reduce(P, splits, ldp, M, N, C, ldc, ctx);
    const cudaError_t f = qgi::scratch_free(ws, ctx);
    return e != cudaSuccess ? e : f;
}

}  // namespace

namespace qgi {

// Any token count: with M <= 128 the second CTA's 128 token rows are zero-filled by the TMA and
// half of each MMA is wasted, but a pair still halves the weight rows each SM dequantises, which
// is what bounds those shapes (measured: 64 x 4096 x 4096 in 23.2 us on pairs against 47.6 us
// on one CTA per 256 weight rows).
bool w4a16_pair_eligible(int M, const qgemm_tensor *W) {
    (void)M;
    return W->rows > BW && W->k % 512 == 0 &&
           reinterpret_cast<uintptr_t>(W->scales) % 16 == 0 && W->lds % 16 == 0;
}

cudaError_t launch_w4a16_pair(const __half *A, int64_t lda, int M, const qgemm_tensor *W,
                              __half *C, int64_t ldc, const LaunchCtx &ctx, bool *encode_ok) {
    return launch_pair_impl<1>(A, lda, M, W, C, ldc, ctx, encode_ok);
}

cudaError_t launch_w4a16_f16s(const __half *A, int64_t lda, int M, const uint8_t *W_int4,
                              int64_t ldw, const __half *scales, int64_t lds_elems, int N, int K,
                              __half *C, int64_t ldc, const LaunchCtx &ctx, bool *encode_ok) {
    qgemm_tensor w{QGEMM_INT4, N, K, W_int4, ldw, reinterpret_cast<const uint8_t *>(scales),
                   lds_elems * 2};
    return launch_pair_impl<2>(A, lda, M, &w, C, ldc, ctx, encode_ok);
}

}  // namespace qgi
