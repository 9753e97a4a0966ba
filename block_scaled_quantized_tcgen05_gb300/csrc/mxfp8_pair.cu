// mxfp8_pair.cu -- block-scaled FP8 and FP4 GEMMs on CTA pairs (tcgen05 cta_group::2).
//
// Same product as mxfp8_gemm.cu (E4M3 data, UE8M0 scale per 32 along K, fp32 accumulation,
// fp16 output), with one MMA spanning two SMs: a cluster of two CTAs computes a 256 x 256 output
// tile; each CTA keeps its own 128 rows of A and its own 128 columns of B in shared memory and
// holds its 128 rows of the accumulator in its TMEM.  Halving the B bytes each SM stages lets six
// stages fit.
//
// Scale factors take two steps.
//  1. sf_pack_kernel rewrites both scale planes into a scratch buffer in the order tcgen05.cp
//     reads them: for each k-tile of 128 and each block of 128 rows, 512 contiguous bytes, 32
//     lines of 16 bytes, line i holding the four scale bytes of rows i, i + 32, i + 64 and i + 96
//     (one 32-bit word per row, byte j = k-block j of the k-tile).  Rows and k-blocks past the
//     operand are written as 0 (scale 2^-127 on zero data).  The row blocks are padded to an even
//     count, so a pair tile never reads past the buffer.
//  2. Each CTA fetches a stage's scales with two 1-D bulk copies (its own 128 rows of A scales,
//     512 bytes; all 256 rows of B scales, 1 KB: contiguous in the repacked layout) onto a barrier
//     of its own, and four scale warps -- one per TMEM lane quarter -- move
//     them from shared memory into this CTA's TMEM with tcgen05.st, in the replicated layout the
//     block-scaled MMA reads (lane 32 q + i, column c: row 32 c + i).  A tcgen05.cp in the MMA
//     stream would sit in the tensor pipe's in-order queue in front of the MMAs; written from
//     registers, the scales never enter that queue.
//
// Hand-off: only the leader (rank 0) issues MMAs; its MMA warp runs the loop and the barrier
// waits together and one elected lane issues (a loop run by one thread alone issues each MMA in
// tens of cycles and leaves the tensor pipe idle between stages).  The loop does one CTA-scope
// barrier wait per stage and nothing else but the four MMAs and a commit.  Each stage's full barrier lives in the leader and
// collects everything the stage needs: the leader's arrival with both CTAs' data bytes, both
// CTAs' data loads, and one arrival from each scale warp of both CTAs once its tcgen05.st have
// completed (tcgen05.wait::st; the arrival itself is relaxed -- a release at cluster scope costs
// about a microsecond per stage).  Commits are multicast to the empty, accumulator-full and drain
// barriers of both CTAs.  Each epilogue warp of both CTAs reads its whole accumulator slice into
// registers first and releases the accumulator with one relaxed arrival on the leader's barrier
// (its TMEM reads are complete at tcgen05.wait::ld), then stores.  Every wait is bounded.
//
// The same pipeline computes the MXFP4 product (E2M1 data packed two per byte, even k in the low
// nibble; the same UE8M0 scale per 32 along K), as kind::mxf4.block_scale.scale_vec::2X MMAs.  A
// stage still moves 128 bytes of each row, now 256 elements: four MMAs of K = 64, each reading two
// scale bytes per row.  The repacked scale lines then come in pairs per stage (W = 2 words per
// row: word w holds k-blocks 4 w .. 4 w + 3 of the stage), and a stage's TMEM slot holds two
// A columns groups and two B column groups.  The kernel is a template over the two formats.
//
// Measured alternatives that lost (or won less): the scales copied by tcgen05.cp from the MMA thread (in this
// kernel the copies serialise with the MMAs once TMA traffic competes for shared memory: +13%);
// scale warps loading the repacked scales from global memory instead of shared memory (+2%);
// direct 16-byte row stores from the epilogue instead of the staged, sector-wide ones (+4%);
// the scale blocks as 2-D tensor boxes 16 bytes wide (+0.6%); raster groups of 8 or 32 pair rows
// instead of 16 (+1%, +5%); L2 prefetch of A and B eight k-tiles ahead (+10%).
#include "qgemm_common.cuh"
#include "qgemm_debug.cuh"
#include "qgemm_internal.h"
#include "qgemm_ptx.cuh"

namespace {

using namespace qg;

constexpr int BM = 128;                     // rows per CTA (256 per pair)
constexpr int BN = 256;                     // columns per pair tile (128 of B per CTA)
constexpr int BK = 128;                     // data bytes of K per stage (128 E4M3, 256 E2M1)
// Warps: 0 producer, 1 MMA issuer, 2..9 epilogue (two per TMEM lane quarter, one per half of
// the 256 accumulator columns, so the accumulator is drained -- and released to the next tile's
// MMAs -- twice as fast as with four), 10..13 scale warps.
constexpr int EPI_WARPS = 8;
constexpr int SCALE_WARP0 = 2 + EPI_WARPS;
constexpr int THREADS = 32 * (SCALE_WARP0 + 4);
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_COL0 = 256;           // scale slots after the 256-column accumulator
constexpr uint32_t A_BYTES = BM * BK;                 // 16 KB
constexpr uint32_t B_BYTES = (BN / 2) * BK;           // 16 KB (this CTA's half)

// Element formats.  W = scale words (4 k-blocks each) per row per stage; one MMA covers W
// k-blocks, so MMA j of a stage reads k-block j W: word (j W) / 4, byte (j W) % 4.
struct FmtE4M3 {
    static constexpr int W = 1;
    static constexpr int ELEMS_PER_BYTE = 1;
    static constexpr int STAGES = 6;
    static constexpr uint32_t SF_COLS_PER_STAGE = 16;   // SFA 4 + SFB 8 (+4 spare)
    // kind::mxf8f6f4 block-scaled descriptor: E4M3 x E4M3 (formats 0), K-major, N = 256,
    // UE8M0 scales, M = 256.
    static constexpr uint32_t IDESC = (static_cast<uint32_t>(BN >> 3) << 17) | (1u << 23) |
                                      (static_cast<uint32_t>(256 >> 7) << 27);
    static __device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                               uint32_t sfa, uint32_t sfb, uint32_t acc) {
        mma_mxf8_pair(d, a, b, idesc, sfa, sfb, acc);
    }
};
struct FmtE2M1 {
    static constexpr int W = 2;
    static constexpr int ELEMS_PER_BYTE = 2;
    static constexpr int STAGES = 5;                    // six do not fit beside 3 KB of scales
    static constexpr uint32_t SF_COLS_PER_STAGE = 24;   // SFA 2 x 4 + SFB 2 x 8
    // kind::mxf4 block-scaled descriptor: E2M1 x E2M1 (format 1 in bits 7-9 and 10-12),
    // K-major, N = 256, UE8M0 scales, M = 256, dense K = 64 (bit 31 clear).
    static constexpr uint32_t IDESC = (1u << 7) | (1u << 10) |
                                      (static_cast<uint32_t>(BN >> 3) << 17) | (1u << 23) |
                                      (static_cast<uint32_t>(256 >> 7) << 27);
    static __device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                               uint32_t sfa, uint32_t sfb, uint32_t acc) {
        mma_mxf4_pair(d, a, b, idesc, sfa, sfb, acc);
    }
};

// Shared-memory map of one format.
template <class F>
struct Smem {
    static constexpr int STAGES = F::STAGES;
    static constexpr uint32_t SFA_BYTES = 512 * F::W;         // 128 rows x 4 W bytes
    static constexpr uint32_t SFB_BYTES = 1024 * F::W;        // 256 rows x 4 W bytes
    static constexpr uint32_t OFF_A = 0;
    static constexpr uint32_t OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr uint32_t OFF_SFA = OFF_B + STAGES * B_BYTES;
    static constexpr uint32_t OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
    static constexpr uint32_t OFF_EPI = OFF_SFB + STAGES * SFB_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_EPI + EPI_WARPS * 2048;
    // full[S] (leader), empty[S], sf_full[S], tmem_full, tmem_empty (leader), drain, then the slot
    static constexpr uint32_t OFF_SLOT = OFF_BAR + (3 * STAGES + 3) * 8;
    static constexpr uint32_t BYTES = OFF_SLOT + 16 + 1024;
    static_assert(BYTES <= 232448, "shared memory budget");
    static_assert(SF_COL0 + STAGES * F::SF_COLS_PER_STAGE <= TMEM_COLS, "TMEM budget");
};

// ------------------------------------------------------------------------ scale repacking
constexpr int PACK_KT = 8;                  // scale words (4 k-blocks) per packing block
constexpr int PACK_ROW = PACK_KT * 4 + 4;   // bytes per staged row (+4 keeps banks apart)

struct SfPackOperand {
    const uint8_t *scales;   // [rows, kcols] UE8M0, row stride lds bytes, any alignment
    int64_t lds;
    int rows;
    int kcols;               // K / 32
    int rbp;                 // padded count of 128-row blocks (even)
    uint8_t *out;            // [KT][rbp][W][32 lines][16 bytes]
    int vec;                 // scales and lds 16-byte aligned: 16-byte loads
};

// grid (max rbp, ceil(KT W / 8), 2 operands) x 256 threads.  Stage 128 rows x 32 scale bytes
// with row-contiguous (coalesced) byte loads, then write 8 scale words x 32 lines of 16 bytes;
// word kw is word kw % W of stage kw / W.
template <int W>
__global__ void __launch_bounds__(256)
sf_pack_kernel(SfPackOperand opA, SfPackOperand opB, int KT, unsigned *err) {
    __shared__ __align__(16) uint8_t tile[128 * PACK_ROW];
    griddep_launch_dependents();   // the GEMM, a programmatic dependent, may start its set-up
    const SfPackOperand &op = blockIdx.z == 0 ? opA : opB;
    const int rb = blockIdx.x;
    if (rb >= op.rbp) return;
    const int kt0 = blockIdx.y * PACK_KT;
    const int t = threadIdx.x;
    if (op.vec && kt0 * 4 + 32 <= op.kcols) {
        // 128 rows x 32 bytes as 256 16-byte loads: thread t takes half t & 1 of row t / 2
        const int row = t >> 1, half = t & 1;
        const int r = rb * 128 + row;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r < op.rows)
            v = __ldg(reinterpret_cast<const uint4 *>(op.scales + static_cast<int64_t>(r) * op.lds +
                                                      kt0 * 4 + 16 * half));
        uint32_t *dst = reinterpret_cast<uint32_t *>(tile + row * PACK_ROW + 16 * half);
        dst[0] = v.x;
        dst[1] = v.y;
        dst[2] = v.z;
        dst[3] = v.w;
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int idx = t + 256 * j;              // 128 rows x 32 bytes
            const int row = idx >> 5, col = idx & 31;
            const int r = rb * 128 + row, c = kt0 * 4 + col;
            uint8_t v = 0;
            if (r < op.rows && c < op.kcols) v = op.scales[static_cast<int64_t>(r) * op.lds + c];
            tile[row * PACK_ROW + col] = v;
        }
    }
    __syncthreads();
    const int ktl = t >> 5, i = t & 31;
    const int kw = kt0 + ktl;
    if (kw >= KT * W) return;
    const uint32_t *w = reinterpret_cast<const uint32_t *>(tile);
    constexpr int WPR = PACK_ROW / 4;             // words per staged row
    uint4 v;
    v.x = w[i * WPR + ktl];
    v.y = w[(i + 32) * WPR + ktl];
    v.z = w[(i + 64) * WPR + ktl];
    v.w = w[(i + 96) * WPR + ktl];
    const int64_t off = (((static_cast<int64_t>(kw / W) * op.rbp + rb) * W + kw % W) * 32 + i) * 16;
    // the repacked plane holds KT x rbp x W x 32 lines of 16 bytes
    if (QG_IN_BOUNDS(err, off >= 0 && off + 16 <= static_cast<int64_t>(KT) * op.rbp * W * 512))
        *reinterpret_cast<uint4 *>(op.out + off) = v;
}

// -------------------------------------------------------------------------------- the GEMM
// K is in data bytes (K elements of E4M3, K / 2 of E2M1).
template <class F>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
mx_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmB64,
               const uint8_t *__restrict__ packA, const uint8_t *__restrict__ packB,
               int rbpA, int rbpB, __half *__restrict__ C, int64_t ldc, int c_vec, int M, int N,
               int K, int epi, unsigned *err, uint64_t timeout_ns) {
    using L = Smem<F>;
    constexpr int STAGES = L::STAGES;
    constexpr int W = F::W;
    constexpr uint32_t SFA_BYTES = L::SFA_BYTES, SFB_BYTES = L::SFB_BYTES;
    constexpr uint32_t OFF_A = L::OFF_A, OFF_B = L::OFF_B, OFF_SFA = L::OFF_SFA,
                       OFF_SFB = L::OFF_SFB, OFF_EPI = L::OFF_EPI, OFF_BAR = L::OFF_BAR,
                       OFF_SLOT = L::OFF_SLOT;
    constexpr uint32_t SF_COLS_PER_STAGE = F::SF_COLS_PER_STAGE;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_1024(smem_raw);
    griddep_launch_dependents();   // a dependent launch (e.g. a clock probe) may run beside
    const uint32_t sb = smem_u32(smem);
    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();      // 0 = leader
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;

    auto full_bar = [&](int s) { return sb + OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sb + OFF_BAR + 8u * (STAGES + s); };
    auto sf_full = [&](int s) { return sb + OFF_BAR + 8u * (2 * STAGES + s); };
    const uint32_t tmem_full = sb + OFF_BAR + 8u * (3 * STAGES);
    const uint32_t tmem_empty = tmem_full + 8;
    const uint32_t drain_bar = tmem_full + 16;
    volatile uint32_t *slot = reinterpret_cast<volatile uint32_t *>(smem + OFF_SLOT);

    const int tiles_m = (M + 2 * BM - 1) / (2 * BM);
    const int tiles_n = (N + BN - 1) / BN;
    const int num_tiles = tiles_m * tiles_n;
    const int KT = (K + BK - 1) / BK;
    const PairWork work(num_tiles, npairs);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 9);   // leader's expect_tx + one lane of each scale warp (x8)
            mbar_init(empty_bar(s), 1);  // leader's multicast commit
            mbar_init(sf_full(s), 1);    // this CTA's scale TMA
        }
        mbar_init(tmem_full, 1);
        mbar_init(tmem_empty, 2 * EPI_WARPS);   // one lane of each epilogue warp of both CTAs
        mbar_init(drain_bar, 1);
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmB64);
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
        // The whole warp runs the loop and waits; one elected lane issues the copies.  The
        // kernel is launched as a programmatic dependent of the scale repack: its set-up above
        // overlaps the repack, and the producer, the only role that reads the repacked scales
        // from global memory (every other role waits on what it loads), waits for it here.
        griddep_wait();
        {
            uint32_t stage = 0, phase = 0;
            int issued = 0;
            bool ok = true;
            const uint64_t keep = l2_policy_evict_last();   // B panels are re-read by many tiles
            for (int it = pair; it < work.n_items && ok; it += npairs) {
                int tile, half, mb, nb;
                work.item(it, tile, half);
                tile_coords(tile, tiles_m, tiles_n, mb, nb);
                const int m0 = mb * 2 * BM + static_cast<int>(rank) * BM;
                const int la = (2 * mb + static_cast<int>(rank)) * 32;   // packed A line
                // a whole tile: 128 B rows per CTA and both 128-row blocks of B scales; a half
                // tile: 64 B rows per CTA and the one block of scales of its 128 columns
                const int nh = half < 0 ? nb * BN + static_cast<int>(rank) * (BN / 2)
                                        : nb * BN + half * (BN / 2) + static_cast<int>(rank) * (BN / 4);
                const int lb = (2 * nb + (half < 0 ? 0 : half)) * 32;     // packed B line
                const uint32_t b_bytes = half < 0 ? B_BYTES : B_BYTES / 2;
                const uint32_t sfb_bytes = half < 0 ? SFB_BYTES : SFB_BYTES / 2;
                for (int kt = 0; kt < KT; ++kt) {
                    if (!mbar_wait_warp(empty_bar(stage), phase ^ 1, timeout_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t lead_full = map_to_cta(full_bar(stage), 0);
                    // debug build: the stage's scale lines lie inside the repacked planes, and
                    // the copies' innermost coordinate is a multiple of 16 bytes
                    const int64_t sa_off = (static_cast<int64_t>(kt) * rbpA * 32 + la) * 16 * W;
                    const int64_t sb_off = (static_cast<int64_t>(kt) * rbpB * 32 + lb) * 16 * W;
                    if (!(QG_IN_BOUNDS(err, (kt * BK) % 16 == 0) &&
                          QG_IN_BOUNDS(err, sa_off >= 0 && sa_off + SFA_BYTES <=
                                                static_cast<int64_t>(KT) * rbpA * 512 * W) &&
                          QG_IN_BOUNDS(err, sb_off >= 0 && sb_off + sfb_bytes <=
                                                static_cast<int64_t>(KT) * rbpB * 512 * W))) {
                        ok = false;
                        break;
                    }
                    if (elect_one()) {
                        if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * (A_BYTES + b_bytes));
                        tma_load_2d_pair(sb + OFF_A + stage * A_BYTES, &tmA, lead_full, kt * BK, m0);
                        tma_load_2d_pair_hint(sb + OFF_B + stage * B_BYTES, half < 0 ? &tmB : &tmB64,
                                              lead_full, kt * BK, nh, keep);
                        mbar_arrive_expect_tx(sf_full(stage), SFA_BYTES + sfb_bytes);
                        bulk_load(sb + OFF_SFA + stage * SFA_BYTES, packA + sa_off, SFA_BYTES,
                                  sf_full(stage));
                        bulk_load(sb + OFF_SFB + stage * SFB_BYTES, packB + sb_off, sfb_bytes,
                                  sf_full(stage));
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
            if (rank == 0)   // the leader's full barriers count both CTAs' loads
                for (int i = max(0, issued - STAGES); i < issued; ++i)
                    if (!__all_sync(0xFFFFFFFFu, mbar_wait_cluster(full_bar(i % STAGES),
                                                                   (i / STAGES) & 1, timeout_ns))) {
                        if (lane == 0) atomicOr(err, ERR_DRAIN);
                        break;
                    }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (rank == 0) {
            // --------------------------------------------------------- MMA issuer
            // The whole warp runs the loop and waits; one elected lane issues.  (A loop run by
            // one lane alone issues measurably slower: the tensor pipe idles between stages.)
            // Descriptors of stage 0; stage s adds s * bytes / 16 to the start-address field.
            const uint64_t adesc0 = smem_desc(sb + OFF_A, 16, 1024, SWZ_128B);
            const uint64_t bdesc0 = smem_desc(sb + OFF_B, 16, 1024, SWZ_128B);
            uint32_t acc_phase = 0, stage = 0, phase = 0;
            bool ok = true;
            for (int it = pair; it < work.n_items && ok; it += npairs) {
                int tile, half;
                work.item(it, tile, half);
                // N = 256, or 128 for a half tile
                const uint32_t idesc = half < 0 ? F::IDESC
                                                : (F::IDESC & ~(0x3Fu << 17)) |
                                                      (static_cast<uint32_t>((BN / 2) >> 3) << 17);
                if (!__all_sync(0xFFFFFFFFu,
                                mbar_wait_cluster(tmem_empty, acc_phase ^ 1, timeout_ns))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kt = 0; kt < KT; ++kt) {
                    if (!mbar_wait_warp(full_bar(stage), phase, timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sf_col = tmem_base + SF_COL0 + stage * SF_COLS_PER_STAGE;
                    const uint64_t adesc = adesc0 + stage * (A_BYTES >> 4);
                    const uint64_t bdesc = bdesc0 + stage * (B_BYTES >> 4);
                    if (elect_one()) {
                        // MMA j: 32 bytes of K at byte 32 j; its first k-block is j W, i.e.
                        // byte (j W) % 4 of scale word (j W) / 4 (SFA word w at +4 w, SFB at
                        // +4 W + 8 w)
#pragma unroll
                        for (uint32_t j = 0; j < BK / 32; ++j) {
                            const uint32_t blk = j * W, w = blk >> 2, id = blk & 3;
                            F::mma(tmem_base, adesc + 2 * j, bdesc + 2 * j,
                                   idesc | (id << 4) | (id << 29), sf_col + 4 * w,
                                   sf_col + 4 * W + 8 * w, (kt > 0 || j > 0) ? 1u : 0u);
                        }
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
    } else if (warp >= SCALE_WARP0) {
        // ------------------------------------------------------------- scale warps
        // Lane i of the warp for lane quarter q writes TMEM lane 32 q + i of the stage's slot:
        // for scale word w, columns 4 w .. 4 w + 3 the A scales of rows i + 32 c and columns
        // 4 W + 8 w .. 4 W + 8 w + 7 the B scales of rows i + 32 c.
        const uint32_t q = warp & 3;
        const uint32_t lead_full = map_to_cta(full_bar(0), 0);
        const int my_items = pair < work.n_items ? (work.n_items - pair + npairs - 1) / npairs : 0;
        const int total = my_items * KT;
        for (int it = 0; it < total; ++it) {
            const uint32_t s = static_cast<uint32_t>(it % STAGES);
            // the TMA of this stage was issued after the MMAs that last read this slot finished
            if (!mbar_wait(sf_full(s), static_cast<uint32_t>(it / STAGES) & 1, timeout_ns)) {
                if (lane == 0) atomicOr(err, ERR_PRODUCER);
                break;
            }
            // shared layout: A [W][32 lines][16], B [2 row blocks][W][32 lines][16]
            const uint8_t *sfa = smem + OFF_SFA + s * SFA_BYTES + lane * 16;
            const uint8_t *sfb = smem + OFF_SFB + s * SFB_BYTES + lane * 16;
            const uint32_t col = tmem_base + ((q * 32) << 16) + SF_COL0 + s * SF_COLS_PER_STAGE;
#pragma unroll
            for (int w = 0; w < W; ++w) {
                const uint4 va = *reinterpret_cast<const uint4 *>(sfa + 512 * w);
                const uint4 vb0 = *reinterpret_cast<const uint4 *>(sfb + 512 * w);
                const uint4 vb1 = *reinterpret_cast<const uint4 *>(sfb + 512 * (W + w));
                tmem_st_32x32b_x4(col + 4 * w, va);
                tmem_st_32x32b_x8(col + 4 * W + 8 * w, vb0, vb1);
            }
            tmem_wait_st();
            tc_fence_before();
            // the slot's scale bytes were read through the generic proxy; its next fill is a TMA write
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive_relaxed_cluster(lead_full + 8u * s);
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const uint32_t q = warp & 3;                     // TMEM lane quarter of this warp
        const uint32_t half = (warp - 2) >> 2;            // accumulator columns [128 h, 128 h + 128)
        const uint32_t lead_empty = map_to_cta(tmem_empty, 0);
        uint32_t acc_phase = 0;
        for (int it = pair; it < work.n_items; it += npairs) {
            int tile, thalf, mb, nb;
            work.item(it, tile, thalf);
            tile_coords(tile, tiles_m, tiles_n, mb, nb);
            if (!mbar_wait_sleep(tmem_full, acc_phase, timeout_ns, 32)) {
                if (lane == 0) atomicOr(err, ERR_EPILOGUE);
                break;
            }
            tc_fence_after();
            const int em0 = mb * 2 * BM + static_cast<int>(rank) * BM;
            const uint32_t stg = sb + OFF_EPI + (warp - 2) * 2048;
            if (thalf < 0) {
                const int en0 = nb * BN + static_cast<int>(half) * (BN / 2);
                if (epi & EPI_ACC_BIT)   // reads the old C: chunk by chunk
                    epilogue_tile<BN / 2, 3>(tmem_base + half * (BN / 2), q, lane, C, ldc, em0,
                                             en0, M, N, c_vec != 0, lead_empty, stg, epi);
                else
                    epilogue_tile_early<BN / 2>(tmem_base + half * (BN / 2), q, lane, C, ldc, em0,
                                                en0, M, N, c_vec != 0, lead_empty, stg,
                                                (epi & EPI_RELU_BIT) != 0);
            } else {
                // a half tile's 128 accumulator columns, 64 per warp of each lane quarter
                const int en0 = nb * BN + thalf * (BN / 2) + static_cast<int>(half) * (BN / 4);
                if (epi & EPI_ACC_BIT)
                    epilogue_tile<BN / 4, 3>(tmem_base + half * (BN / 4), q, lane, C, ldc, em0,
                                             en0, M, N, c_vec != 0, lead_empty, stg, epi);
                else
                    epilogue_tile_early<BN / 4>(tmem_base + half * (BN / 4), q, lane, C, ldc, em0,
                                                en0, M, N, c_vec != 0, lead_empty, stg,
                                                (epi & EPI_RELU_BIT) != 0);
            }
            acc_phase ^= 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();                   // no remote arrival or multicast targets an exited CTA
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

int padded_blocks(int64_t rows) { return static_cast<int>(2 * ((rows + 255) / 256)); }

// Data bytes of K for a view of format F (K elements).
template <class F>
int64_t k_bytes(const qgemm_tensor *t) { return t->k / F::ELEMS_PER_BYTE; }

template <class F>
size_t pair_scratch_bytes(const qgemm_tensor *A, const qgemm_tensor *B) {
    const int64_t KT = (k_bytes<F>(A) + BK - 1) / BK;
    return static_cast<size_t>(KT) * (padded_blocks(A->rows) + padded_blocks(B->rows)) * 512 *
           F::W;
}

template <class F>
SfPackOperand pack_operand(const qgemm_tensor *t, uint8_t *out) {
    const int vec = (reinterpret_cast<uintptr_t>(t->scales) % 16 == 0 && t->lds % 16 == 0) ? 1 : 0;
    return SfPackOperand{t->scales, t->lds, static_cast<int>(t->rows), static_cast<int>(t->k / 32),
                         padded_blocks(t->rows), out, vec};
}

// Repack one or two operands' scale planes (nops = 1: opA only).
template <class F>
cudaError_t launch_sf_pack(const SfPackOperand &pa, const SfPackOperand &pb, int nops, int KT,
                           cudaStream_t stream, unsigned *err) {
    const int rbp = nops == 2 && pb.rbp > pa.rbp ? pb.rbp : pa.rbp;
    const dim3 pgrid(static_cast<unsigned>(rbp),
                     static_cast<unsigned>((KT * F::W + PACK_KT - 1) / PACK_KT),
                     static_cast<unsigned>(nops));
    sf_pack_kernel<F::W><<<pgrid, 256, 0, stream>>>(pa, nops == 2 ? pb : pa, KT, err);
    return cudaGetLastError();
}

// The CTA-pair GEMM on scale planes already repacked into packA / packB.
template <class F>
cudaError_t launch_pair_packed(const qgemm_tensor *A, const qgemm_tensor *B, __half *C,
                               int64_t ldc, const uint8_t *packA, const uint8_t *packB,
                               const qgi::LaunchCtx &ctx, bool *encode_ok) {
    const int M = static_cast<int>(A->rows), N = static_cast<int>(B->rows);
    const int Kb = static_cast<int>(k_bytes<F>(A));
    const int rbpA = padded_blocks(M), rbpB = padded_blocks(N);
    CUtensorMap tmA, tmB, tmB64;
    *encode_ok =
        qgi::encode_tma_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A->data, Kb, M, A->ld, BK, BM,
                           CU_TENSOR_MAP_SWIZZLE_128B) &&
        qgi::encode_tma_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B->data, Kb, N, B->ld, BK, BN / 2,
                           CU_TENSOR_MAP_SWIZZLE_128B) &&
        qgi::encode_tma_2d(&tmB64, CU_TENSOR_MAP_DATA_TYPE_UINT8, B->data, Kb, N, B->ld, BK, BN / 4,
                           CU_TENSOR_MAP_SWIZZLE_128B);
    if (!*encode_ok) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(mx_pair_kernel<F>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Smem<F>::BYTES);
    if (e != cudaSuccess) return e;
    const int tiles = ((M + 2 * BM - 1) / (2 * BM)) * ((N + BN - 1) / BN);
    int pairs = ctx.num_sms / 2;
    if (pairs > tiles) pairs = tiles;
    const int c_vec = (reinterpret_cast<uintptr_t>(C) % 16 == 0 && ldc % 8 == 0) ? 1 : 0;
    // a programmatic dependent of the kernel ahead on the stream (the scale repack): it starts
    // once the repack's CTAs have all begun and waits for its results before reading them
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = Smem<F>::BYTES;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];   // the cluster shape is the kernel's own (__cluster_dims__)
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mx_pair_kernel<F>, tmA, tmB, tmB64, packA, packB, rbpA, rbpB,
                              C, ldc, c_vec, M, N, Kb, ctx.epi, ctx.err, ctx.timeout_ns);
}

template <class F>
cudaError_t launch_pair(const qgemm_tensor *A, const qgemm_tensor *B, __half *C, int64_t ldc,
                        void *scratch, const qgi::LaunchCtx &ctx, bool *encode_ok) {
    const int KT = static_cast<int>((k_bytes<F>(A) + BK - 1) / BK);
    uint8_t *packA = static_cast<uint8_t *>(scratch);
    uint8_t *packB = packA + static_cast<size_t>(KT) * padded_blocks(A->rows) * 512 * F::W;
    *encode_ok = true;
    cudaError_t e = launch_sf_pack<F>(pack_operand<F>(A, packA), pack_operand<F>(B, packB), 2,
                                      KT, ctx.stream, ctx.err);
    if (e != cudaSuccess) return e;
    return launch_pair_packed<F>(A, B, C, ldc, packA, packB, ctx, encode_ok);
}

}  // namespace

namespace qgi {

bool mxfp8_pair_eligible(const qgemm_tensor *A, const qgemm_tensor *B) {
    return A->rows > BM && B->rows > BN / 2;
}

size_t mxfp8_pair_scratch_bytes(const qgemm_tensor *A, const qgemm_tensor *B) {
    return pair_scratch_bytes<FmtE4M3>(A, B);
}

cudaError_t launch_mxfp8_pair(const qgemm_tensor *A, const qgemm_tensor *B, __half *C,
                              int64_t ldc, void *scratch, const LaunchCtx &ctx, bool *encode_ok) {
    return launch_pair<FmtE4M3>(A, B, C, ldc, scratch, ctx, encode_ok);
}

size_t mxfp8_pack_bytes(const qgemm_tensor *T) {
    const int64_t KT = (k_bytes<FmtE4M3>(T) + BK - 1) / BK;
    return static_cast<size_t>(KT) * padded_blocks(T->rows) * 512 * FmtE4M3::W;
}

cudaError_t launch_mxfp8_sf_pack(const qgemm_tensor *T, void *out, const LaunchCtx &ctx) {
    const int KT = static_cast<int>((k_bytes<FmtE4M3>(T) + BK - 1) / BK);
    const SfPackOperand op = pack_operand<FmtE4M3>(T, static_cast<uint8_t *>(out));
    return launch_sf_pack<FmtE4M3>(op, op, 1, KT, ctx.stream, ctx.err);
}

cudaError_t launch_mxfp8_pair_packed(const qgemm_tensor *A, const qgemm_tensor *B, __half *C,
                                     int64_t ldc, const void *packA, const void *packB,
                                     const LaunchCtx &ctx, bool *encode_ok) {
    return launch_pair_packed<FmtE4M3>(A, B, C, ldc, static_cast<const uint8_t *>(packA),
                                       static_cast<const uint8_t *>(packB), ctx, encode_ok);
}

size_t mxfp4_scratch_bytes(const qgemm_tensor *A, const qgemm_tensor *B) {
    return pair_scratch_bytes<FmtE2M1>(A, B);
}

cudaError_t launch_mxfp4_pair(const qgemm_tensor *A, const qgemm_tensor *B, __half *C,
                              int64_t ldc, void *scratch, const LaunchCtx &ctx, bool *encode_ok) {
    return launch_pair<FmtE2M1>(A, B, C, ldc, scratch, ctx, encode_ok);
}

}  // namespace qgi
