// f16_gemm.cu -- fp16 GEMM on tcgen05 (kind::f16, fp32 accumulation in TMEM, fp16 output).
//
// C[M, N] = fp16_rn(A[M, K] @ B[K, N]); A row-major (K-major operand), B row-major [K, N]
// (N contiguous: an MN-major operand).  The unquantized half x half -> half matmul of
// "TensorOps: quantized matmul ..." (kernel M0 of "VALIDATED ON M4 MAX") and of the TileLang
// page's fast path (fp16 in, fp32 accumulate, cast to fp16 on store), on GB300's pipeline:
//   warp 0     producer: per 64-wide k-tile one TMA box of A (128 rows x 128 B) and BN/64
//              boxes of B (64 k-rows x 64 n = 128 B), all with the 128-byte swizzle.
//   warp 1     TMEM owner + MMA issuer: four 128 x BN x 16 MMAs per k-tile; B is described
//              as MN-major (64-element swizzle atoms BN/64 apart, 8-row k groups 1 KB apart).
//   warps 2-5  epilogue: TMEM -> fp16 -> global, masked at the M / N edges (or, when K is split
//              over several CTAs because there are few tiles, TMEM -> an fp32 partial plane that
//              splitk_reduce.cu adds in order).
// Shapes with more than one 128-row and one 128-column block use the CTA-pair kernel below.
#include "qgemm_common.cuh"
#include "qgemm_debug.cuh"
#include "qgemm_internal.h"
#include "qgemm_ptx.cuh"

#include <algorithm>

namespace {

using namespace qg;

constexpr int BM = 128;
constexpr int BK = 64;         // fp16 elements of K per k-tile (one 128-byte swizzle row)
constexpr int THREADS = 192;
constexpr int SPLIT_UNIT = 8;  // split-K ranges are whole 512-wide slices of K (8 k-tiles)


template <int BN>
struct Cfg {
    static constexpr int STAGES = (BN == 256) ? 4 : 6;
    static constexpr uint32_t A_BYTES = BM * BK * 2;      // 16 KB
    static constexpr uint32_t B_ATOM_BYTES = BK * 64 * 2; // 64 k-rows x 64 n = 8 KB
    static constexpr uint32_t B_BYTES = (BN / 64) * B_ATOM_BYTES;
    static constexpr uint32_t OFF_A = 0;
    static constexpr uint32_t OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr uint32_t OFF_EPI = OFF_B + STAGES * B_BYTES;   // 4 warps x 2 KB
    static constexpr uint32_t OFF_BAR = OFF_EPI + 4 * 2048;
    static constexpr uint32_t OFF_SLOT = OFF_BAR + (2 * STAGES + 5) * 8;
    static constexpr uint32_t TMEM_COLS = 2 * BN <= 256 ? 256 : 512;   // two accumulators
    static constexpr uint32_t SMEM_BYTES = OFF_SLOT + 16 + 1024;
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B fp16 (format 0),
// A K-major (bit 15 = 0), B MN-major (bit 16 = 1), N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t f16_idesc(int n) {
    return (1u << 4) | (1u << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(BM >> 4) << 24);
}

template <int BN>
__global__ void __launch_bounds__(THREADS, 1)
gemm_f16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                __half *__restrict__ C, int64_t ldc, int c_vec, int M, int N, int K, int splits,
                float *__restrict__ P, int64_t ldp, int epi, unsigned *err, uint64_t timeout_ns) {
    using G = Cfg<BN>;
    constexpr int S = G::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_1024(smem_raw);
    // a kernel launched after this one as a programmatic dependent (a decode GEMV, the split-K
    // reduction) may be scheduled now: it waits for this grid's completion before it touches
    // memory, and its launch no longer waits for the last CTA to exit
    griddep_launch_dependents();
    const uint32_t sb = smem_u32(smem);
    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;

    auto full_bar = [&](int s) { return sb + G::OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sb + G::OFF_BAR + 8u * (S + s); };
    // accumulator double buffer: tmem_full[2], tmem_empty[2], then the drain barrier
    const uint32_t acc_bar0 = sb + G::OFF_BAR + 8u * (2 * S);
    auto tmem_full = [&](uint32_t b) { return acc_bar0 + 8u * b; };
    auto tmem_empty = [&](uint32_t b) { return acc_bar0 + 16u + 8u * b; };
    const uint32_t drain_bar = acc_bar0 + 32;
    volatile uint32_t *slot = reinterpret_cast<volatile uint32_t *>(smem + G::OFF_SLOT);

    const int tiles_m = (M + BM - 1) / BM;
    const int tiles_n = (N + BN - 1) / BN;
    const int num_tiles = tiles_m * tiles_n;
    const int num_items = num_tiles * splits;        // (tile, k range) work items
    const int KT = (K + BK - 1) / BK;
    const int64_t plane = static_cast<int64_t>(M) * ldp;   // floats per split-K partial plane

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(tmem_full(0), 1);
        mbar_init(tmem_full(1), 1);
        mbar_init(tmem_empty(0), 128);             // every epilogue thread
        mbar_init(tmem_empty(1), 128);
        mbar_init(drain_bar, 1);
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(const_cast<uint32_t *>(slot)), G::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *slot;

    if (warp == 0) {
        uint32_t stage = 0, phase = 0;
        int issued = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < num_items && ok; it += gridDim.x) {
            int tile, split, kt0, kt1, mb, nb;
            split_item(it, num_tiles, splits, KT, SPLIT_UNIT, tile, split, kt0, kt1);
            tile_coords(tile, tiles_m, tiles_n, mb, nb);
            for (int kt = kt0; kt < kt1; ++kt) {
                if (!mbar_wait(empty_bar(stage), phase ^ 1, timeout_ns)) {
                    ok = false;
                    break;
                }
                // debug build: the copies' innermost coordinates are multiples of 16 bytes
                if (!QG_IN_BOUNDS(err, (kt * BK) % 8 == 0 && (nb * BN) % 8 == 0)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t sA = sb + G::OFF_A + stage * G::A_BYTES;
                    const uint32_t sB = sb + G::OFF_B + stage * G::B_BYTES;
                    mbar_arrive_expect_tx(full_bar(stage), G::A_BYTES + G::B_BYTES);
                    tma_load_2d(sA, &tmA, full_bar(stage), kt * BK, mb * BM);
#pragma unroll
                    for (int c = 0; c < BN / 64; ++c)
                        tma_load_2d(sB + c * G::B_ATOM_BYTES, &tmB, full_bar(stage),
                                    nb * BN + 64 * c, kt * BK);
                }
                __syncwarp();
                ++issued;
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        if (!ok && lane == 0) atomicOr(err, ERR_PRODUCER);
        for (int i = max(0, issued - S); i < issued; ++i) {
            if (!mbar_wait(full_bar(i % S), (i / S) & 1, timeout_ns)) {
                if (lane == 0) atomicOr(err, ERR_DRAIN);
                break;
            }
        }
    } else if (warp == 1) {
        // MMA issuer: the whole warp runs the loop and its waits, one elected lane issues, the
        // descriptors computed outside the issuing branch (stage s adds s * bytes / 16 to the
        // start-address field).  MN-major B: LBO = stride between 64-wide N atoms, SBO = 8 k-rows.
        const uint64_t adesc0 = smem_desc(sb + G::OFF_A, 16, 1024, SWZ_128B);
        const uint64_t bdesc0 = smem_desc(sb + G::OFF_B, G::B_ATOM_BYTES, 1024, SWZ_128B);
        uint32_t stage = 0, phase = 0, acc_it = 0;
        bool ok = true;
        const uint32_t idesc = f16_idesc(BN);
        for (int it = blockIdx.x; it < num_items && ok; it += gridDim.x) {
            int tile, split, kt0, kt1;
            split_item(it, num_tiles, splits, KT, SPLIT_UNIT, tile, split, kt0, kt1);
            const uint32_t ab = acc_it & 1;       // accumulator buffer of this item
            if (!mbar_wait_warp(tmem_empty(ab), ((acc_it >> 1) & 1) ^ 1, timeout_ns)) {
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
                const uint64_t adesc = adesc0 + stage * (G::A_BYTES >> 4);
                const uint64_t bdesc = bdesc0 + stage * (G::B_BYTES >> 4);
                if (elect_one()) {
#pragma unroll
                    for (uint32_t j = 0; j < BK / 16; ++j) {
                        // A: 16 halves = 32 bytes along the swizzle row; B: 16 k-rows = 2 KB
                        mma_f16(tmem_base + ab * BN, adesc + 2 * j, bdesc + 128 * j, idesc,
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
        if (elect_one()) {
            if (!ok) atomicOr(err, ERR_MMA);
            tc_commit(drain_bar);
        }
        __syncwarp();
        if (!mbar_wait(drain_bar, 0, timeout_ns) && lane == 0) atomicOr(err, ERR_DRAIN);
    } else {
        const uint32_t q = warp & 3;
        uint32_t acc_it = 0;
        for (int it = blockIdx.x; it < num_items; it += gridDim.x) {
            int tile, split, kt0, kt1, mb, nb;
            split_item(it, num_tiles, splits, KT, SPLIT_UNIT, tile, split, kt0, kt1);
            tile_coords(tile, tiles_m, tiles_n, mb, nb);
            const uint32_t ab = acc_it & 1;
            if (!mbar_wait_sleep(tmem_full(ab), (acc_it >> 1) & 1, timeout_ns, 128)) {
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
    if (warp == 1) tmem_dealloc(tmem_base, G::TMEM_COLS);
}

template <int BN>
cudaError_t launch_bn(const __half *A, int64_t lda, const __half *B, int64_t ldb, __half *C,
                      int64_t ldc, int M, int N, int K, int splits, float *P, int64_t ldp,
                      const qgi::LaunchCtx &ctx, bool *encode_ok) {
    using G = Cfg<BN>;
    CUtensorMap tmA, tmB;
    *encode_ok = qgi::encode_tma_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, K, M, lda * 2, BK,
                                    BM, CU_TENSOR_MAP_SWIZZLE_128B) &&
                 qgi::encode_tma_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, B, N, K, ldb * 2, 64,
                                    BK, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!*encode_ok) return cudaErrorInvalidValue;
    auto kern = gemm_f16_kernel<BN>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int64_t items = static_cast<int64_t>((M + BM - 1) / BM) * ((N + BN - 1) / BN) * splits;
    const int grid = items < ctx.num_sms ? static_cast<int>(items) : ctx.num_sms;
    const int c_vec = (reinterpret_cast<uintptr_t>(C) % 16 == 0 && ldc % 8 == 0) ? 1 : 0;
    kern<<<grid, THREADS, G::SMEM_BYTES, ctx.stream>>>(tmA, tmB, C, ldc, c_vec, M, N, K, splits, P,
                                                        ldp, ctx.epi, ctx.err, ctx.timeout_ns);
    return cudaGetLastError();
}

// Split-K on the one-CTA route, as for the one-CTA MXFP8 GEMM: when the output has at most half
// as many tiles as the GPU has SMs, each tile's k-tiles are shared out over up to SMs / tiles CTAs
// (whole 512-wide slices of K), which write fp32 partial planes (M rows of tiles_n * BN floats)
// that splitk_reduce.cu adds in split order.
int f16_splits(int M, int N, int K, int bn, int num_sms) {
    const int64_t tiles = static_cast<int64_t>((M + BM - 1) / BM) * ((N + bn - 1) / bn);
    const int64_t units = ((K + BK - 1) / BK + SPLIT_UNIT - 1) / SPLIT_UNIT;
    if (2 * tiles > num_sms) return 1;
    const int64_t s = std::min<int64_t>(num_sms / tiles, units);
    return s < 1 ? 1 : static_cast<int>(s);
}

template <int BN>
cudaError_t launch_one_cta(const __half *A, int64_t lda, const __half *B, int64_t ldb, __half *C,
                           int64_t ldc, int M, int N, int K, const qgi::LaunchCtx &ctx,
                           bool *encode_ok) {
    const int splits = f16_splits(M, N, K, BN, ctx.num_sms);
    const int64_t ldp = static_cast<int64_t>((N + BN - 1) / BN) * BN;
    void *ws = nullptr;
    if (splits > 1) {
        const cudaError_t e = qgi::scratch_alloc(
            static_cast<size_t>(splits) * static_cast<size_t>(M) * static_cast<size_t>(ldp) * sizeof(float),
            ctx, &ws);
        if (e != cudaSuccess) return e;
    }
    float *P = static_cast<float *>(ws);
    cudaError_t e = launch_bn<BN>(A, lda, B, ldb, C, ldc, M, N, K, splits, P, ldp, ctx, encode_ok);
    if (e == cudaSuccess && splits > 1) e = qgi::launch_splitk_reduce(P, splits, ldp, M, N, C, ldc, ctx);
    const cudaError_t f = qgi::scratch_free(ws, ctx);
    return e != cudaSuccess ? e : f;
}

// ------------------------------------------------------------------------------------------
// CTA-pair variant (tcgen05 cta_group::2): a cluster of two CTAs computes a 256 x 256 tile; each
// CTA stages its own 128 rows of A and 128 columns of B (six stages fit) and holds its 128
// accumulator rows in TMEM (two accumulators).  The leader (rank 0) arms each stage's full
// barrier with both CTAs' bytes and issues the MMAs; its commits are multicast to both CTAs'
// barriers; one lane per epilogue warp of both CTAs releases an accumulator on the leader.
// Last wave: when the tiles left after the last full wave of pairs fit twice into one wave, each
// of them is computed as two 256 x 128 halves (N = 128 MMAs, one 64-column B box per CTA) by two
// pairs, so the last wave takes half a tile's time instead of a whole one (4096^3: 256 tiles on 76
// pairs are 3.37 waves; this way 3.5 tile times instead of 4).
constexpr int P_BM = 128;       // rows per CTA (the pair covers 256)
constexpr int P_BN = 256;       // columns per pair tile (128 stored per CTA)
constexpr int P_BK = 64;
constexpr int P_STAGES = 6;
constexpr int P_THREADS = 192;
constexpr uint32_t P_TMEM_COLS = 512;      // two 256-column accumulators
constexpr uint32_t P_A_BYTES = P_BM * P_BK * 2;          // 16 KB
constexpr uint32_t P_B_ATOM = P_BK * 64 * 2;           // 8 KB
constexpr uint32_t P_B_BYTES = 2 * P_B_ATOM;           // this CTA's 128 columns
constexpr uint32_t P_OFF_A = 0;
constexpr uint32_t P_OFF_B = P_OFF_A + P_STAGES * P_A_BYTES;
constexpr uint32_t P_OFF_EPI = P_OFF_B + P_STAGES * P_B_BYTES;
constexpr uint32_t P_OFF_BAR = P_OFF_EPI + 4 * 2048;
// full[S] (leader), empty[S], tmem_full[2], tmem_empty[2] (leader), drain
constexpr uint32_t P_OFF_SLOT = P_OFF_BAR + (2 * P_STAGES + 5) * 8;
constexpr uint32_t P_SMEM_BYTES = P_OFF_SLOT + 16 + 1024;
static_assert(P_SMEM_BYTES <= 232448, "smem");

// kind::f16, D fp32, A K-major, B MN-major, N = 256 (or 128 for a half tile), M = 256 (pair)
constexpr uint32_t P_IDESC = (1u << 4) | (1u << 16) | (static_cast<uint32_t>(P_BN >> 3) << 17) |
                           (static_cast<uint32_t>(256 >> 4) << 24);
constexpr uint32_t P_IDESC_HALF = (1u << 4) | (1u << 16) | (static_cast<uint32_t>((P_BN / 2) >> 3) << 17) |
                                (static_cast<uint32_t>(256 >> 4) << 24);

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(P_THREADS, 1)
gemm_f16_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     __half *__restrict__ C, int64_t ldc, int c_vec, int M, int N, int K,
                     int epi, unsigned *err, uint64_t timeout_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_1024(smem_raw);
    // a kernel launched after this one as a programmatic dependent (a decode GEMV) may be
    // scheduled now: it waits for this grid's completion before it touches memory, and its
    // launch no longer waits for the last CTA to exit
    griddep_launch_dependents();
    const uint32_t sb = smem_u32(smem);
    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();          // 0 = leader (issues the MMAs)
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;

    auto full_bar = [&](int s) { return sb + P_OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sb + P_OFF_BAR + 8u * (P_STAGES + s); };
    const uint32_t acc_bar0 = sb + P_OFF_BAR + 8u * (2 * P_STAGES);
    auto tmem_full = [&](uint32_t b) { return acc_bar0 + 8u * b; };
    auto tmem_empty = [&](uint32_t b) { return acc_bar0 + 16u + 8u * b; };
    const uint32_t drain_bar = acc_bar0 + 32;
    volatile uint32_t *slot = reinterpret_cast<volatile uint32_t *>(smem + P_OFF_SLOT);

    const int tiles_m = (M + 2 * P_BM - 1) / (2 * P_BM);
    const int tiles_n = (N + P_BN - 1) / P_BN;
    const int num_tiles = tiles_m * tiles_n;
    const int KT = (K + P_BK - 1) / P_BK;
    const PairWork work(num_tiles, npairs);

    if (threadIdx.x == 0) {
        for (int s = 0; s < P_STAGES; ++s) {
            mbar_init(full_bar(s), 1);     // the leader's expect_tx for both CTAs' bytes
            mbar_init(empty_bar(s), 1);    // the leader's multicast commit
        }
        mbar_init(tmem_full(0), 1);
        mbar_init(tmem_full(1), 1);
        mbar_init(tmem_empty(0), 8);       // one lane of each epilogue warp of both CTAs
        mbar_init(tmem_empty(1), 8);
        mbar_init(drain_bar, 1);
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(const_cast<uint32_t *>(slot)), P_TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();                        // peer barriers initialised before any remote use
    tc_fence_after();
    const uint32_t tmem_base = *slot;

    if (warp == 0) {
        // producer: the whole warp runs the loop and waits; one elected lane issues the copies
        {
            uint32_t stage = 0, phase = 0;
            int issued = 0;
            bool ok = true;
            for (int it = pair; it < work.n_items && ok; it += npairs) {
                int tile, half, mb, nb;
                work.item(it, tile, half);
                tile_coords(tile, tiles_m, tiles_n, mb, nb);
                const int m0 = mb * 2 * P_BM + static_cast<int>(rank) * P_BM;
                // a whole tile: 128 columns per CTA; a half tile: 64 columns per CTA
                const int nh = half < 0 ? nb * P_BN + static_cast<int>(rank) * (P_BN / 2)
                                        : nb * P_BN + half * (P_BN / 2) + static_cast<int>(rank) * 64;
                const uint32_t tx = 2 * (P_A_BYTES + (half < 0 ? P_B_BYTES : P_B_ATOM));
                for (int kt = 0; kt < KT; ++kt) {
                    if (!mbar_wait_warp(empty_bar(stage), phase ^ 1, timeout_ns)) {
                        ok = false;
                        break;
                    }
                    // debug build: the copies' innermost coordinates are multiples of 16 bytes
                    if (!QG_IN_BOUNDS(err, (kt * P_BK) % 8 == 0 && nh % 8 == 0)) {
                        ok = false;
                        break;
                    }
                    const uint32_t lead_full = map_to_cta(full_bar(stage), 0);
                    if (elect_one()) {
                        if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), tx);
                        const uint32_t sA = sb + P_OFF_A + stage * P_A_BYTES;
                        const uint32_t sB = sb + P_OFF_B + stage * P_B_BYTES;
                        tma_load_2d_pair(sA, &tmA, lead_full, kt * P_BK, m0);
                        tma_load_2d_pair(sB, &tmB, lead_full, nh, kt * P_BK);
                        if (half < 0)
                            tma_load_2d_pair(sB + P_B_ATOM, &tmB, lead_full, nh + 64, kt * P_BK);
                    }
                    __syncwarp();
                    ++issued;
                    if (++stage == P_STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok && lane == 0) atomicOr(err, ERR_PRODUCER);
            if (rank == 0)   // the leader's full barriers count both CTAs' bytes
                for (int i = max(0, issued - P_STAGES); i < issued; ++i)
                    if (!__all_sync(0xFFFFFFFFu,
                                    mbar_wait_cluster(full_bar(i % P_STAGES), (i / P_STAGES) & 1,
                                                      timeout_ns))) {
                        if (lane == 0) atomicOr(err, ERR_DRAIN);
                        break;
                    }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (rank == 0) {
            // MMA issuer: the whole warp runs the loop and its waits, one elected lane issues.
            // Descriptors of stage 0; stage s adds s * bytes / 16 to the start-address field.
            const uint64_t adesc0 = smem_desc(sb + P_OFF_A, 16, 1024, SWZ_128B);
            const uint64_t bdesc0 = smem_desc(sb + P_OFF_B, P_B_ATOM, 1024, SWZ_128B);
            uint32_t stage = 0, phase = 0, acc_it = 0;
            bool ok = true;
            for (int it = pair; it < work.n_items && ok; it += npairs) {
                int tile, half;
                work.item(it, tile, half);
                const uint32_t idesc = half < 0 ? P_IDESC : P_IDESC_HALF;
                const uint32_t ab = acc_it & 1;
                if (!__all_sync(0xFFFFFFFFu, mbar_wait_cluster(tmem_empty(ab),
                                                               ((acc_it >> 1) & 1) ^ 1, timeout_ns))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kt = 0; kt < KT; ++kt) {
                    // CTA scope: the stage's bytes arrive on this barrier by TMA from both CTAs
                    if (!mbar_wait_warp(full_bar(stage), phase, timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = adesc0 + stage * (P_A_BYTES >> 4);
                    const uint64_t bdesc = bdesc0 + stage * (P_B_BYTES >> 4);
                    if (elect_one()) {
#pragma unroll
                        for (uint32_t j = 0; j < P_BK / 16; ++j)
                            mma_f16_pair(tmem_base + ab * P_BN, adesc + 2 * j, bdesc + 128 * j, idesc,
                                         (kt > 0 || j > 0) ? 1u : 0u);
                        tc_commit_pair(empty_bar(stage), 3);
                    }
                    __syncwarp();
                    if (++stage == P_STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                if (elect_one()) tc_commit_pair(tmem_full(ab), 3);
                __syncwarp();
                ++acc_it;
            }
            if (elect_one()) {
                if (!ok) atomicOr(err, ERR_MMA);
                tc_commit_pair(drain_bar, 3);
            }
            __syncwarp();
        }
        // both CTAs: every pair MMA writing this CTA's TMEM has completed
        if (!mbar_wait(drain_bar, 0, timeout_ns) && lane == 0) atomicOr(err, ERR_DRAIN);
    } else {
        const uint32_t q = warp & 3;
        uint32_t acc_it = 0;
        for (int it = pair; it < work.n_items; it += npairs) {
            int tile, half, mb, nb;
            work.item(it, tile, half);
            tile_coords(tile, tiles_m, tiles_n, mb, nb);
            const uint32_t ab = acc_it & 1;
            if (!mbar_wait_sleep(tmem_full(ab), (acc_it >> 1) & 1, timeout_ns, 128)) {
                if (lane == 0) atomicOr(err, ERR_EPILOGUE);
                break;
            }
            tc_fence_after();
            const int m0 = mb * 2 * P_BM + static_cast<int>(rank) * P_BM;
            if (half < 0)
                epilogue_tile<P_BN, 2>(tmem_base + ab * P_BN, q, lane, C, ldc, m0, nb * P_BN, M, N,
                                       c_vec != 0, map_to_cta(tmem_empty(ab), 0),
                                       sb + P_OFF_EPI + (warp - 2) * 2048, epi);
            else
                epilogue_tile<P_BN / 2, 2>(tmem_base + ab * P_BN, q, lane, C, ldc, m0,
                                           nb * P_BN + half * (P_BN / 2), M, N, c_vec != 0,
                                           map_to_cta(tmem_empty(ab), 0),
                                           sb + P_OFF_EPI + (warp - 2) * 2048, epi);
            ++acc_it;
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();                        // no remote arrival or multicast targets an exited CTA
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, P_TMEM_COLS);
}

}  // namespace

namespace qgi {

static cudaError_t launch_gemm_f16_pair(const __half *A, int64_t lda, const __half *B,
                                        int64_t ldb, __half *C, int64_t ldc, int M, int N, int K,
                                        const LaunchCtx &ctx, bool *encode_ok) {
    CUtensorMap tmA, tmB;
    *encode_ok = encode_tma_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, K, M, lda * 2, P_BK, P_BM,
                               CU_TENSOR_MAP_SWIZZLE_128B) &&
                 encode_tma_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, B, N, K, ldb * 2, 64, P_BK,
                               CU_TENSOR_MAP_SWIZZLE_128B);
    if (!*encode_ok) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gemm_f16_pair_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int tiles = ((M + 2 * P_BM - 1) / (2 * P_BM)) * ((N + P_BN - 1) / P_BN);
    int pairs = ctx.num_sms / 2;
    if (pairs > tiles) pairs = tiles;
    const int c_vec = (reinterpret_cast<uintptr_t>(C) % 16 == 0 && ldc % 8 == 0) ? 1 : 0;
    gemm_f16_pair_kernel<<<2 * pairs, P_THREADS, P_SMEM_BYTES, ctx.stream>>>(
        tmA, tmB, C, ldc, c_vec, M, N, K, ctx.epi, ctx.err, ctx.timeout_ns);
    return cudaGetLastError();
}

cudaError_t launch_gemm_f16(const __half *A, int64_t lda, const __half *B, int64_t ldb,
                            __half *C, int64_t ldc, int M, int N, int K, const LaunchCtx &ctx,
                            bool *encode_ok) {
    // CTA pairs once there are at least two 128-row blocks and more than one 128-column block.
    if (M > 128 && N > 128)
        return launch_gemm_f16_pair(A, lda, B, ldb, C, ldc, M, N, K, ctx, encode_ok);
    if (N > 128) return launch_one_cta<256>(A, lda, B, ldb, C, ldc, M, N, K, ctx, encode_ok);
    return launch_one_cta<128>(A, lda, B, ldb, C, ldc, M, N, K, ctx, encode_ok);
}

}  // namespace qgi
