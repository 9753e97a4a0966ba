// w4a16_gemm.cu -- weight-only int4 GEMM for prefill shapes on tcgen05.
//
// C[M, N] = fp16_rn( sum_k A[m, k] * q(W[n, k]) * 2^(SW[n, k/32] - 127) ),  fp32 accumulation.
//
// "TensorOps: quantized matmul ..." (sections "Revised kernel strategy" and "M2 = block-32 fp16
// scaling") dequantises each 32-block of int4 weights with its scale into on-chip memory and
// then runs the half x half matmul; the same page's escape-hatch note recommends dequantising
// straight into the operand the matrix unit reads.  On GB300 the operand the tensor core reads
// is shared memory in the 128-byte-swizzled K-major layout, so converter warps write the
// dequantised fp16 weight tile directly in that layout:
//   warp 0     TMA producer for the activation tile A (128 rows x 64 k, 128-byte swizzle).
//   warp 1     TMEM owner + MMA issuer (kind::f16, both operands K-major).
//   warps 2-5  epilogue (TMEM -> fp16 -> global).
//   warps 6-13 converters: cp.async the packed int4 bytes and scale words of future k-tiles into
//              a private ring (each thread consumes only what it copied), then per 32-block
//              turn 32 nibbles into fp16 (q + 8 placed in the mantissa of 1024, minus 1032; the
//              high nibble as 1024 + 16 (q + 8), times 1/16, minus 72), multiply by the fp16
//              power of two 2^(e-127) and store 16-byte chunks at their swizzled position.
// The fp16 weight q * 2^(e-127) is exact for 103 <= e <= 139; other bytes give 0 (NaN for 255)
// and the rows where that matters are rewritten by w4a16_outlier.cu (w4a16_convert.cuh).
#include "qgemm_common.cuh"
#include "qgemm_debug.cuh"
#include "qgemm_internal.h"
#include "qgemm_ptx.cuh"
#include "w4a16_convert.cuh"

namespace {

using namespace qg;

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int RAW = 3;            // k-tiles of int4 prefetched ahead by each converter thread
constexpr int CONV_THREADS = 256;
constexpr int THREADS = 192 + CONV_THREADS;
constexpr uint32_t TMEM_COLS = 512;   // two 256-column accumulators
constexpr int UNITS = 2;          // (row, 32-block) units per converter thread per k-tile

constexpr uint32_t A_BYTES = BM * BK * 2;
constexpr uint32_t B_BYTES = BN * BK * 2;
constexpr uint32_t RAW_DATA_BYTES = UNITS * CONV_THREADS * 16;  // [unit][thread] 16 B
constexpr uint32_t RAW_SCALE_BYTES = UNITS * CONV_THREADS * 4;  // [unit][thread] 4 B
constexpr uint32_t RAW_SLOT_BYTES = RAW_DATA_BYTES + RAW_SCALE_BYTES;
constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = OFF_A + STAGES * A_BYTES;
constexpr uint32_t OFF_RAW = OFF_B + STAGES * B_BYTES;
constexpr uint32_t OFF_BAR = OFF_RAW + RAW * RAW_SLOT_BYTES;
constexpr uint32_t OFF_SLOT = OFF_BAR + (2 * STAGES + 5) * 8;
constexpr uint32_t OFF_FLAGS = OFF_SLOT + 16;   // [2][BN] outlier-column flags (accumulate)
constexpr uint32_t SMEM_BYTES = OFF_FLAGS + 2 * BN + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// kind::f16, D fp32, A and B fp16, both K-major, N = 256, M = 128.
constexpr uint32_t IDESC = (1u << 4) | (static_cast<uint32_t>(BN >> 3) << 17) |
                           (static_cast<uint32_t>(BM >> 4) << 24);

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_4_full(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---- accumulate epilogue with outlier rows --------------------------------------------------
// When the output is accumulated (C = relu?(A W^T + C_old)), the columns of outlier weight rows
// (w4_row_is_outlier) are neither read nor written here: w4a16_outlier_kernel computes them from
// the old C afterwards.  The four epilogue warps mark the tile's 256 weight rows in shared memory
// (flags[c] != 0: skip column n0 + c) before the tile's accumulator is ready.
__device__ __forceinline__ void mark_outlier_cols(uint8_t *flags, int t, int n0, int N, int K,
                                                  const uint8_t *W, int64_t ldw,
                                                  const uint8_t *SW, int64_t ldsw) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int c = t + 128 * h;
        const int n = n0 + c;
        flags[c] = (n < N && w4_row_is_outlier(SW + static_cast<int64_t>(n) * ldsw,
                                               W + static_cast<int64_t>(n) * ldw, K / 32))
                       ? 1 : 0;
    }
}

// Barrier of the four epilogue warps (named barrier 2, 128 threads) that also ANDs `ok` over
// them: every epilogue thread reaches it once per tile, so a wait that ran out in one warp
// stops all four together.
__device__ __forceinline__ bool epi_bar_and(bool ok) {
    uint32_t all_ok;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(all_ok)
        : "r"(ok ? 1u : 0u)
        : "memory");
    return all_ok != 0;
}

// Drain one 128 x BN accumulator with C = relu?(acc + C_old), skipping flagged columns (element
// stores; used only for tiles that hold an outlier column).  Every lane arrives on tmem_empty
// after the last TMEM read, as epilogue_tile does.
__device__ __forceinline__ void epilogue_acc_masked(uint32_t tmem_base, uint32_t q, uint32_t lane,
                                                    __half *C, int64_t ldc, int m0, int n0, int M,
                                                    int N, uint32_t tmem_empty, int epi,
                                                    const uint8_t *flags) {
    const int row = m0 + static_cast<int>(q * 32 + lane);
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ++ch) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_base + ((q * 32) << 16) + ch * 32, v);
        tmem_wait_ld();
        if (ch == BN / 32 - 1) {
            tc_fence_before();
            mbar_arrive(tmem_empty);
        }
        const uint32_t skip = __ballot_sync(0xFFFFFFFFu, flags[ch * 32 + lane] != 0);
        if (row >= M) continue;
        __half *crow = C + static_cast<int64_t>(row) * ldc;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int col = n0 + ch * 32 + i;
            if (col < N && !((skip >> i) & 1u)) {
                float x = __uint_as_float(v[i]) + __half2float(crow[col]);
                if (epi & EPI_RELU_BIT) x = fmaxf(x, 0.0f);
                crow[col] = __float2half_rn(x);
            }
        }
    }
}

template <bool SF_VEC>
__global__ void __launch_bounds__(THREADS, 1)
w4a16_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const uint8_t *__restrict__ W,
                  int64_t ldw, const uint8_t *__restrict__ SW, int64_t ldsw,
                  __half *__restrict__ C, int64_t ldc, int c_vec, int M, int N, int K, int epi,
                  unsigned *err,
                  uint64_t timeout_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_1024(smem_raw);
    griddep_launch_dependents();   // the outlier-row pass may take the room this CTA leaves
    const uint32_t sb = smem_u32(smem);
    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;

    auto full_bar = [&](int s) { return sb + OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sb + OFF_BAR + 8u * (STAGES + s); };
    // accumulator double buffer: tmem_full[2], tmem_empty[2], then the drain barrier
    const uint32_t acc_bar0 = sb + OFF_BAR + 8u * (2 * STAGES);
    auto tmem_full = [&](uint32_t b) { return acc_bar0 + 8u * b; };
    auto tmem_empty = [&](uint32_t b) { return acc_bar0 + 16u + 8u * b; };
    const uint32_t drain_bar = acc_bar0 + 32;
    volatile uint32_t *slot = reinterpret_cast<volatile uint32_t *>(smem + OFF_SLOT);

    const int tiles_m = (M + BM - 1) / BM;
    const int tiles_n = (N + BN - 1) / BN;
    const int num_tiles = tiles_m * tiles_n;
    const int KT = K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1 + CONV_THREADS);  // TMA arrival + every converter thread
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(tmem_full(0), 1);
        mbar_init(tmem_full(1), 1);
        mbar_init(tmem_empty(0), 128);             // every epilogue thread
        mbar_init(tmem_empty(1), 128);
        mbar_init(drain_bar, 1);
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
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
        // -------------------------------------------------------- activation producer
        uint32_t stage = 0, phase = 0;
        int issued = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
            int mb, nb;
            tile_coords(tile, tiles_m, tiles_n, mb, nb);
            for (int kt = 0; kt < KT; ++kt) {
                if (!mbar_wait(empty_bar(stage), phase ^ 1, timeout_ns)) {
                    ok = false;
                    break;
                }
                // debug build: the copies' innermost coordinates are multiples of 16 bytes
                if (!QG_IN_BOUNDS(err, (kt * BK) % 8 == 0)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(full_bar(stage), A_BYTES);
                    tma_load_2d(sb + OFF_A + stage * A_BYTES, &tmA, full_bar(stage), kt * BK,
                                mb * BM);
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
            if (!mbar_wait(full_bar(i % STAGES), (i / STAGES) & 1, timeout_ns)) {
                if (lane == 0) atomicOr(err, ERR_DRAIN);
                break;
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        // The whole warp runs the loop and its waits, one elected lane issues; descriptors of
        // stage 0 computed once, stage s adding s * bytes / 16 to the start-address field.
        const uint64_t adesc0 = smem_desc(sb + OFF_A, 16, 1024, SWZ_128B);
        const uint64_t bdesc0 = smem_desc(sb + OFF_B, 16, 1024, SWZ_128B);
        uint32_t stage = 0, phase = 0, acc_it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
            const uint32_t ab = acc_it & 1;       // accumulator buffer of this tile
            if (!mbar_wait_warp(tmem_empty(ab), ((acc_it >> 1) & 1) ^ 1, timeout_ns)) {
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
                const uint64_t adesc = adesc0 + stage * (A_BYTES >> 4);
                const uint64_t bdesc = bdesc0 + stage * (B_BYTES >> 4);
                if (elect_one()) {
#pragma unroll
                    for (uint32_t j = 0; j < BK / 16; ++j)
                        mma_f16(tmem_base + ab * BN, adesc + 2 * j, bdesc + 2 * j, IDESC,
                                (kt > 0 || j > 0) ? 1u : 0u);
                    tc_commit(empty_bar(stage));
                }
                __syncwarp();
                if (++stage == STAGES) {
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
    } else if (warp < 6) {
        // ------------------------------------------------------------------- epilogue
        const uint32_t q = warp & 3;
        const bool acc_mode = (epi & EPI_ACC_BIT) != 0;
        uint32_t acc_it = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            int mb, nb;
            tile_coords(tile, tiles_m, tiles_n, mb, nb);
            const uint32_t ab = acc_it & 1;
            uint8_t *flags = smem + OFF_FLAGS + ab * BN;
            if (acc_mode)
                mark_outlier_cols(flags, static_cast<int>(threadIdx.x) - 64, nb * BN, N, K, W, ldw,
                                  SW, ldsw);
            bool got = mbar_wait_sleep(tmem_full(ab), (acc_it >> 1) & 1, timeout_ns, 128);
            if (acc_mode) got = epi_bar_and(got);
            if (!got) {
                if (lane == 0) atomicOr(err, ERR_EPILOGUE);
                break;
            }
            tc_fence_after();
            bool masked = false;
            if (acc_mode) {
#pragma unroll
                for (int c = 0; c < BN / 32; ++c)
                    masked |= __any_sync(0xFFFFFFFFu, flags[c * 32 + lane] != 0);
            }
            if (masked)
                epilogue_acc_masked(tmem_base + ab * BN, q, lane, C, ldc, mb * BM, nb * BN, M, N,
                                    tmem_empty(ab), epi, flags);
            else
                epilogue_tile<BN>(tmem_base + ab * BN, q, lane, C, ldc, mb * BM, nb * BN, M, N,
                                  c_vec != 0, tmem_empty(ab), 0u, epi);
            ++acc_it;
        }
    } else {
        // ----------------------------------------------------------------- converters
        const int ct = static_cast<int>(threadIdx.x) - 192;   // 0..CONV_THREADS-1
        const int h = ct & 1;                                   // which 32-block of the k-tile
        const int rsub = ct >> 1;                               // row within each row group
        constexpr int ROW_STEP = CONV_THREADS / 2;              // rows between a thread's units
        const int my_tiles = (num_tiles > static_cast<int>(blockIdx.x))
                                 ? (num_tiles - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1
                                 : 0;
        const int total = my_tiles * KT;
        // k-tiles are issued and consumed in order: tile and k index kept as running counters
        int iss_tile = static_cast<int>(blockIdx.x), iss_kt = 0, iss_mb = 0, iss_nb = 0;
        if (total > 0) tile_coords(iss_tile, tiles_m, tiles_n, iss_mb, iss_nb);
        auto issue = [&](int it) {
            if (it < total) {
                const int kt = iss_kt;
                const int nb = iss_nb;
                const uint32_t rs = sb + OFF_RAW + (it % RAW) * RAW_SLOT_BYTES;
                const int blk = kt * 2 + h;                     // scale block index along K
#pragma unroll
                for (int i = 0; i < UNITS; ++i) {
                    int n = nb * BN + ROW_STEP * i + rsub;
                    n = n < N ? n : N - 1;                      // rows past N are never stored
                    const uint8_t *src = W + static_cast<int64_t>(n) * ldw + kt * (BK / 2) + 16 * h;
                    cp_async_16(rs + (i * CONV_THREADS + ct) * 16, src);
                    if constexpr (SF_VEC) {
                        // the aligned scale word holding this block's byte
                        const uint8_t *ssrc = SW + static_cast<int64_t>(n) * ldsw + (blk & ~3);
                        cp_async_4_full(rs + RAW_DATA_BYTES + (i * CONV_THREADS + ct) * 4, ssrc);
                    }
                }
                if (++iss_kt == KT) {
                    iss_kt = 0;
                    iss_tile += static_cast<int>(gridDim.x);
                    if (it + 1 < total) tile_coords(iss_tile, tiles_m, tiles_n, iss_mb, iss_nb);
                }
            }
            cp_async_commit();
        };
#pragma unroll
        for (int p = 0; p < RAW; ++p) issue(p);
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        int kt = 0, cur_tile = static_cast<int>(blockIdx.x), mb_cur = 0, nb_cur = 0;
        if (!SF_VEC && total > 0) tile_coords(cur_tile, tiles_m, tiles_n, mb_cur, nb_cur);
        for (int it = 0; it < total; ++it) {
            cp_async_wait<RAW - 1>();
            if (!mbar_wait(empty_bar(stage), phase ^ 1, timeout_ns)) {
                ok = false;
                break;
            }
            const uint8_t *rs = smem + OFF_RAW + (it % RAW) * RAW_SLOT_BYTES;
            const uint32_t sB = sb + OFF_B + stage * B_BYTES;
            const int blk = kt * 2 + h;
#pragma unroll
            for (int i = 0; i < UNITS; ++i) {
                const uint4 d = *reinterpret_cast<const uint4 *>(rs + (i * CONV_THREADS + ct) * 16);
                uint32_t e;
                if constexpr (SF_VEC) {
                    const uint32_t sw = *reinterpret_cast<const uint32_t *>(
                        rs + RAW_DATA_BYTES + (i * CONV_THREADS + ct) * 4);
                    e = (sw >> (8 * (blk & 3))) & 0xFF;
                } else {
                    int n = nb_cur * BN + ROW_STEP * i + rsub;
                    n = n < N ? n : N - 1;
                    e = __ldg(SW + static_cast<int64_t>(n) * ldsw + blk);
                }
                const int r = ROW_STEP * i + rsub;               // row inside the 256-row tile
                const uint32_t words[4] = {d.x, d.y, d.z, d.w};
                const bool fast = fused_ok(e);
                uint32_t s2, c2;
                if (fast) fused_consts(e, s2, c2);
                else s2 = ue8m0_to_f16x2(e);
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    uint32_t o[4];
                    if (fast) i4x8_to_f16_fused(words[w], s2, c2, o);
                    else i4x8_to_f16(words[w], s2, o);
                    const int c = 4 * h + w;                     // 16-byte chunk (8 k) in the row
                    const uint32_t dst = sB + r * 128 + ((c ^ (r & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(o[0]),
                                 "r"(o[1]), "r"(o[2]), "r"(o[3])
                                 : "memory");
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(full_bar(stage));
            issue(it + RAW);
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1;
            }
            if (++kt == KT) {
                kt = 0;
                cur_tile += static_cast<int>(gridDim.x);
                if (!SF_VEC && it + 1 < total) tile_coords(cur_tile, tiles_m, tiles_n, mb_cur, nb_cur);
            }
        }
        cp_async_wait<0>();
        if (!ok && lane == 0) atomicOr(err, ERR_PRODUCER);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// ------------------------------------------------------------------------------------------
// TMA-fed variant (weights and scale rows 16-byte aligned).  The producer also loads the packed
// int4 tile of each k-tile (256 rows x 32 bytes, into the last 8 KB of that stage's fp16 B
// buffer) and, every 8 k-tiles, the 16 scale bytes per row that cover them (into one of two
// staging slots).  Converter threads read their two (row, 32-block) units and scale bytes from
// shared memory, meet at a named barrier (all packed bytes read before anyone overwrites the
// buffer), then write the dequantised fp16 tile over the whole buffer.
constexpr int T_CONV = 256;
constexpr int T_THREADS = 192 + T_CONV;
constexpr int T_UNITS = 2;
constexpr int T_SF_GROUP = 8;                          // k-tiles per 16-byte scale group
constexpr uint32_t T_RAW_BYTES = BN * (BK / 2);        // 8 KB packed int4 per k-tile
constexpr uint32_t T_RAW_OFF = B_BYTES - T_RAW_BYTES;  // inside the stage's B buffer
constexpr uint32_t T_STG = BN * 16;                    // 4 KB scale group
constexpr uint32_t T_OFF_STG = OFF_B + STAGES * B_BYTES;
constexpr uint32_t T_OFF_EPI = T_OFF_STG + 2 * T_STG;   // 4 epilogue warps x 2 KB
constexpr uint32_t T_OFF_BAR = T_OFF_EPI + 4 * 2048;
// raw_full[S], conv_full[S], empty[S], tmem_full[2], tmem_empty[2], drain, then the TMEM slot
constexpr uint32_t T_OFF_SLOT = T_OFF_BAR + (3 * STAGES + 5) * 8;
constexpr uint32_t T_OFF_FLAGS = T_OFF_SLOT + 16;
constexpr uint32_t T_SMEM_BYTES = T_OFF_FLAGS + 2 * BN + 1024;
static_assert(T_SMEM_BYTES <= 232448, "shared memory budget");

__global__ void __launch_bounds__(T_THREADS, 1)
w4a16_tma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                 const __grid_constant__ CUtensorMap tmS, const uint8_t *__restrict__ W,
                 int64_t ldw, const uint8_t *__restrict__ SW, int64_t ldsw,
                 __half *__restrict__ C, int64_t ldc,
                 int c_vec, int M, int N, int K, int epi, unsigned *err, uint64_t timeout_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_1024(smem_raw);
    griddep_launch_dependents();   // the outlier-row pass may take the room this CTA leaves
    const uint32_t sb = smem_u32(smem);
    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;

    auto raw_full = [&](int s) { return sb + T_OFF_BAR + 8u * s; };
    auto conv_full = [&](int s) { return sb + T_OFF_BAR + 8u * (STAGES + s); };
    auto empty_bar = [&](int s) { return sb + T_OFF_BAR + 8u * (2 * STAGES + s); };
    // accumulator double buffer: tmem_full[2], tmem_empty[2], then the drain barrier
    const uint32_t acc_bar0 = sb + T_OFF_BAR + 8u * (3 * STAGES);
    auto tmem_full = [&](uint32_t b) { return acc_bar0 + 8u * b; };
    auto tmem_empty = [&](uint32_t b) { return acc_bar0 + 16u + 8u * b; };
    const uint32_t drain_bar = acc_bar0 + 32;
    volatile uint32_t *slot = reinterpret_cast<volatile uint32_t *>(smem + T_OFF_SLOT);

    const int tiles_m = (M + BM - 1) / BM;
    const int tiles_n = (N + BN - 1) / BN;
    const int num_tiles = tiles_m * tiles_n;
    const int KT = K / BK;
    const int ngk = (KT + T_SF_GROUP - 1) / T_SF_GROUP;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(raw_full(s), 1);          // producer's expect_tx arrival
            mbar_init(conv_full(s), T_CONV);    // every converter thread
            mbar_init(empty_bar(s), 1);         // tcgen05.commit
        }
        mbar_init(tmem_full(0), 1);
        mbar_init(tmem_full(1), 1);
        mbar_init(tmem_empty(0), 128);             // every epilogue thread
        mbar_init(tmem_empty(1), 128);
        mbar_init(drain_bar, 1);
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmS);
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
        // ------------------------------------------- producer: A, packed W, scale groups
        uint32_t stage = 0, phase = 0;
        int issued = 0;
        bool ok = true;
        int tile_iter = 0;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++tile_iter) {
            int mb, nb;
            tile_coords(tile, tiles_m, tiles_n, mb, nb);
            for (int kt = 0; kt < KT; ++kt) {
                if (!mbar_wait(empty_bar(stage), phase ^ 1, timeout_ns)) {
                    ok = false;
                    break;
                }
                // debug build: the copies' innermost coordinates are multiples of 16 bytes
                if (!QG_IN_BOUNDS(err, (kt * BK) % 8 == 0 && (kt * (BK / 2)) % 16 == 0 && (16 * (kt / T_SF_GROUP)) % 8 == 0)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const bool grp = (kt % T_SF_GROUP) == 0;
                    const int q = tile_iter * ngk + kt / T_SF_GROUP;
                    const uint32_t sB = sb + OFF_B + stage * B_BYTES;
                    mbar_arrive_expect_tx(raw_full(stage),
                                          A_BYTES + T_RAW_BYTES + (grp ? T_STG : 0u));
                    tma_load_2d(sb + OFF_A + stage * A_BYTES, &tmA, raw_full(stage), kt * BK,
                                mb * BM);
                    tma_load_2d(sB + T_RAW_OFF, &tmW, raw_full(stage), kt * (BK / 2), nb * BN);
                    if (grp)
                        tma_load_2d(sb + T_OFF_STG + (q & 1) * T_STG, &tmS, raw_full(stage),
                                    16 * (kt / T_SF_GROUP), nb * BN);
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
            if (!mbar_wait(raw_full(i % STAGES), (i / STAGES) & 1, timeout_ns)) {
                if (lane == 0) atomicOr(err, ERR_DRAIN);
                break;
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        // The whole warp runs the loop and its waits, one elected lane issues; descriptors of
        // stage 0 computed once, stage s adding s * bytes / 16 to the start-address field.
        const uint64_t adesc0 = smem_desc(sb + OFF_A, 16, 1024, SWZ_128B);
        const uint64_t bdesc0 = smem_desc(sb + OFF_B, 16, 1024, SWZ_128B);
        uint32_t stage = 0, phase = 0, acc_it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
            const uint32_t ab = acc_it & 1;       // accumulator buffer of this tile
            if (!mbar_wait_warp(tmem_empty(ab), ((acc_it >> 1) & 1) ^ 1, timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            for (int kt = 0; kt < KT; ++kt) {
                if (!mbar_wait_warp(raw_full(stage), phase, timeout_ns) ||
                    !mbar_wait_warp(conv_full(stage), phase, timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t adesc = adesc0 + stage * (A_BYTES >> 4);
                const uint64_t bdesc = bdesc0 + stage * (B_BYTES >> 4);
                if (elect_one()) {
#pragma unroll
                    for (uint32_t j = 0; j < BK / 16; ++j)
                        mma_f16(tmem_base + ab * BN, adesc + 2 * j, bdesc + 2 * j, IDESC,
                                (kt > 0 || j > 0) ? 1u : 0u);
                    tc_commit(empty_bar(stage));
                }
                __syncwarp();
                if (++stage == STAGES) {
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
    } else if (warp < 6) {
        // ------------------------------------------------------------------- epilogue
        const uint32_t q = warp & 3;
        const bool acc_mode = (epi & EPI_ACC_BIT) != 0;
        uint32_t acc_it = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            int mb, nb;
            tile_coords(tile, tiles_m, tiles_n, mb, nb);
            const uint32_t ab = acc_it & 1;
            uint8_t *flags = smem + T_OFF_FLAGS + ab * BN;
            if (acc_mode)
                mark_outlier_cols(flags, static_cast<int>(threadIdx.x) - 64, nb * BN, N, K, W, ldw,
                                  SW, ldsw);
            bool got = mbar_wait_sleep(tmem_full(ab), (acc_it >> 1) & 1, timeout_ns, 128);
            if (acc_mode) got = epi_bar_and(got);
            if (!got) {
                if (lane == 0) atomicOr(err, ERR_EPILOGUE);
                break;
            }
            tc_fence_after();
            bool masked = false;
            if (acc_mode) {
#pragma unroll
                for (int c = 0; c < BN / 32; ++c)
                    masked |= __any_sync(0xFFFFFFFFu, flags[c * 32 + lane] != 0);
            }
            if (masked)
                epilogue_acc_masked(tmem_base + ab * BN, q, lane, C, ldc, mb * BM, nb * BN, M, N,
                                    tmem_empty(ab), epi, flags);
            else
                epilogue_tile<BN>(tmem_base + ab * BN, q, lane, C, ldc, mb * BM, nb * BN, M, N,
                                  c_vec != 0, tmem_empty(ab), sb + T_OFF_EPI + (warp - 2) * 2048,
                                  epi);
            ++acc_it;
        }
    } else {
        // ----------------------------------------------------------------- converters
        const int ct = static_cast<int>(threadIdx.x) - 192;     // 0 .. T_CONV-1
        const int h = ct & 1;                                     // 32-block of the k-tile
        const int rsub = ct >> 1;                                 // rows rsub, rsub + 128
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        int tile_iter = 0;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++tile_iter) {
            for (int kt = 0; kt < KT; ++kt) {
                const bool got = mbar_wait(raw_full(stage), phase, timeout_ns);
                const int qg = tile_iter * ngk + kt / T_SF_GROUP;
                const uint8_t *stg = smem + T_OFF_STG + (qg & 1) * T_STG;
                const uint8_t *bufp = smem + OFF_B + stage * B_BYTES;
                const int sbyte = (kt % T_SF_GROUP) * 2 + h;     // scale byte within the group
                uint4 d[T_UNITS];
                uint32_t e[T_UNITS];
#pragma unroll
                for (int i = 0; i < T_UNITS; ++i) {
                    const int r = rsub + 128 * i;
                    if (got) {
                        d[i] = *reinterpret_cast<const uint4 *>(bufp + T_RAW_OFF + r * 32 + 16 * h);
                        e[i] = stg[r * 16 + sbyte];
                    }
                }
                // Every converter has its packed bytes before the buffer is overwritten.  All of
                // them always reach this barrier; if any wait ran out, all of them stop.
                uint32_t all_ok;
                asm volatile(
                    "{\n\t.reg .pred p, q;\n\t"
                    "setp.ne.u32 p, %1, 0;\n\t"
                    "bar.red.and.pred q, 1, %2, p;\n\t"
                    "selp.u32 %0, 1, 0, q;\n\t}"
                    : "=r"(all_ok)
                    : "r"(got ? 1u : 0u), "n"(T_CONV)
                    : "memory");
                if (!all_ok) {
                    ok = false;
                    break;
                }
                const uint32_t sB = sb + OFF_B + stage * B_BYTES;
#pragma unroll
                for (int i = 0; i < T_UNITS; ++i) {
                    const int r = rsub + 128 * i;
                    const bool fast = fused_ok(e[i]);
                    uint32_t s2, c2 = 0;
                    if (fast) fused_consts(e[i], s2, c2);
                    else s2 = ue8m0_to_f16x2(e[i]);
                    const uint32_t words[4] = {d[i].x, d[i].y, d[i].z, d[i].w};
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        uint32_t o[4];
                        if (fast) i4x8_to_f16_fused(words[w], s2, c2, o);
                        else i4x8_to_f16(words[w], s2, o);
                        const int c = 4 * h + w;
                        const uint32_t dst = sB + r * 128 + ((c ^ (r & 7)) << 4);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst),
                                     "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3])
                                     : "memory");
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(conv_full(stage));
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        if (!ok && lane == 0) atomicOr(err, ERR_PRODUCER);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

}  // namespace

namespace qgi {

cudaError_t launch_w4a16(const __half *A, int64_t lda, int M, const qgemm_tensor *W, __half *C,
                         int64_t ldc, const LaunchCtx &ctx, bool *encode_ok) {
    // CTA pairs with the weights dequantised into TMEM when the shape allows (w4a16_pair.cu)
    if (w4a16_pair_eligible(M, W)) return launch_w4a16_pair(A, lda, M, W, C, ldc, ctx, encode_ok);
    const int N = static_cast<int>(W->rows), K = static_cast<int>(W->k);
    CUtensorMap tmA;
    *encode_ok = encode_tma_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, K, M, lda * 2, BK, BM,
                               CU_TENSOR_MAP_SWIZZLE_128B);
    if (!*encode_ok) return cudaErrorInvalidValue;
    const int tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const int grid = tiles < ctx.num_sms ? tiles : ctx.num_sms;
    const int c_vec = (reinterpret_cast<uintptr_t>(C) % 16 == 0 && ldc % 8 == 0) ? 1 : 0;
    // TMA route: 16-byte aligned scale rows and whole 8-k-tile scale groups (K % 512 == 0), so a
    // staging slot is never refilled while converters still read it.
    if (reinterpret_cast<uintptr_t>(W->scales) % 16 == 0 && W->lds % 16 == 0 && K % 512 == 0) {
        CUtensorMap tmW, tmS;
        *encode_ok = encode_tma_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, W->data, K / 2, N, W->ld,
                                   BK / 2, BN, CU_TENSOR_MAP_SWIZZLE_NONE) &&
                     encode_tma_2d(&tmS, CU_TENSOR_MAP_DATA_TYPE_UINT8, W->scales, K / 32, N,
                                   W->lds, 16, BN, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (!*encode_ok) return cudaErrorInvalidValue;
        cudaError_t e = cudaFuncSetAttribute(w4a16_tma_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             T_SMEM_BYTES);
        if (e != cudaSuccess) return e;
        w4a16_tma_kernel<<<grid, T_THREADS, T_SMEM_BYTES, ctx.stream>>>(
            tmA, tmW, tmS, W->data, W->ld, W->scales, W->lds, C, ldc, c_vec, M, N, K, ctx.epi,
            ctx.err, ctx.timeout_ns);
        return cudaGetLastError();
    }
    const bool sf_vec = reinterpret_cast<uintptr_t>(W->scales) % 4 == 0 && W->lds % 4 == 0;
    auto kern = sf_vec ? w4a16_gemm_kernel<true> : w4a16_gemm_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kern<<<grid, THREADS, SMEM_BYTES, ctx.stream>>>(tmA, W->data, W->ld, W->scales, W->lds, C,
                                                    ldc, c_vec, M, N, K, ctx.epi, ctx.err,
                                                    ctx.timeout_ns);
    return cudaGetLastError();
}

}  // namespace qgi
