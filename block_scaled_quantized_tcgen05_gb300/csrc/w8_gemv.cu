// w8_gemv.cu -- decode GEMV with block-scaled int8 weights, bound by HBM bandwidth.
//
// Y[m, n] = fp16_rn( sum_b 2^(SW[n,b]-127) * sum_{k in block b} X[m,k] * W[n,k] ),  M <= 16.
//
// Decode reads every weight byte once, so the kernel is a weight stream ("TensorOps: quantized
// matmul ...", section "Why this matters here": decode is memory-bandwidth-bound and int8
// weights are read at int8 cost).  At M = 16 the arithmetic (2 * 16 flops per weight byte) is
// beyond the fp32 CUDA cores at HBM speed, so the products run on the tensor cores with warp-level
// mma.m16n8k16 (fp16 in, fp32 accumulate), weights as the 16-row operand and the activations as
// the 8-column operand (swap-AB).
//
// Streaming: a producer warp keeps S stages in flight, each one TMA box of 64 weight rows x 128
// bytes of K plus the matching 128-wide slice of X, both with the 128-byte swizzle so that the
// consumers' fragment reads from shared memory are free of bank conflicts.  Four consumer warps
// own 16 weight rows each.  Per 32-element block a lane quad (t = 0..3) takes 8 consecutive
// int8 of rows g and g+8, converts them exactly to fp16 with a byte-permute into the mantissa of
// 1024 (a published integer-to-half technique), and feeds two k16 MMAs; the 32 k of a block are
// permuted identically for weights and activations, so the dot product is unchanged.  The
// block's fp32 partial sum is scaled by 2^(e-127) (exact) and added to the running fp32 sum, so
// every UE8M0 scale is handled exactly.  CTAs are persistent over 64-row blocks.
#include <cuda_fp16.h>

#include "qgemm_common.cuh"
#include "qgemm_internal.h"
#include "qgemm_ptx.cuh"

namespace {

using namespace qg;

constexpr int CONSUMERS = 4;
constexpr int THREADS = (CONSUMERS + 1) * 32;
constexpr int ROWS = CONSUMERS * 16;        // weight rows per CTA iteration
constexpr int KC = 128;                     // K per stage (bytes of int8)
constexpr int STAGES = 6;
constexpr int SCALE_AHEAD = 3;              // scale words prefetched this many chunks ahead

template <int NH>
struct GCfg {
    static constexpr uint32_t W_BYTES = ROWS * KC;            // 8 KB
    static constexpr uint32_t X_HALF = 8 * NH * 128;          // one 64-wide half of the X slice
    static constexpr uint32_t X_BYTES = 2 * X_HALF;
    static constexpr uint32_t STAGE = W_BYTES + X_BYTES;
    static constexpr uint32_t OFF_BAR = STAGES * STAGE;
    static constexpr uint32_t SMEM = OFF_BAR + 2 * STAGES * 8 + 1024;
};

// 4 int8 (one 32-bit word) -> two fp16x2 holding the exact integers (q0,q1), (q2,q3).
__device__ __forceinline__ void i8x4_to_f16x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;                       // q + 128, as unsigned bytes
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x5140u);  // halves 0x64|b0, 0x64|b1
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x5342u);  // halves 0x64|b2, 0x64|b3
    const uint32_t bias = 0x64806480u;                        // 1152.0 = 1024 + 128
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias));
}

// Not volatile: a pure function of its registers, so the compiler may interleave the MMAs of
// independent 32-blocks.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1, const float (&c)[4]) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
          "f"(c[2]), "f"(c[3]));
}

// Four scale bytes (blocks 4c .. 4c+3 of a row) as one little-endian word; bytes past the row's
// last block read as 127 (2^0; their data is zero-filled).
__device__ __forceinline__ uint32_t scale_word(const uint8_t *row, int c, int nblk, bool vec) {
    const int b0 = 4 * c;
    if (vec && b0 + 4 <= nblk) return __ldg(reinterpret_cast<const uint32_t *>(row + b0));
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w |= static_cast<uint32_t>(b0 + i < nblk ? __ldg(row + b0 + i) : 127) << (8 * i);
    return w;
}

// True if some byte of w is 0x00 or 0xFF (the scale codes the shift decode does not cover).
__device__ __forceinline__ bool has_special_byte(uint32_t w) {
    const uint32_t z = (w - 0x01010101u) & ~w & 0x80808080u;     // a zero byte
    const uint32_t n = ~w;
    const uint32_t f = (n - 0x01010101u) & ~n & 0x80808080u;     // a 0xFF byte
    return (z | f) != 0u;
}

// 2^(byte b of w - 127) as fp32 for bytes 1..254: the byte moved into the exponent field.
template <int B>
__device__ __forceinline__ float scale_fast(uint32_t w) {
    const uint32_t bits = (B < 3 ? (w << (23 - 8 * B)) : (w >> 1)) & 0x7F800000u;
    return __uint_as_float(bits);
}

// One 64-row x 128-k stage: four 32-blocks, each two MMAs per activation half, the block's fp32
// partial sum scaled by its power of two.
template <int NH, bool EXACT>
__device__ __forceinline__ void consume_stage(float (&acc)[NH][4], const uint8_t *st,
                                              const uint8_t *xs, int r0, uint32_t sw, int g, int t,
                                              uint32_t e0w, uint32_t e1w) {
    using G = GCfg<NH>;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        // weights: bytes 32 b + 8 t .. +8 of rows r0, r0 + 8 (16-byte chunk 2b + t/2)
        const uint32_t wc = ((static_cast<uint32_t>(2 * b + (t >> 1)) ^ sw) << 4) +
                            static_cast<uint32_t>((t & 1) * 8);
        const uint2 wa = *reinterpret_cast<const uint2 *>(st + r0 * 128 + wc);
        const uint2 wb = *reinterpret_cast<const uint2 *>(st + (r0 + 8) * 128 + wc);
        // activations: halves 32 b + 8 t .. +8 of X rows g (and g + 8)
        const uint8_t *xhalf = xs + static_cast<uint32_t>(b >> 1) * G::X_HALF;
        const uint32_t xc = static_cast<uint32_t>(4 * (b & 1) + t);
        const uint32_t xo = (xc ^ static_cast<uint32_t>(g & 7)) << 4;
        const uint4 xa = *reinterpret_cast<const uint4 *>(xhalf + g * 128 + xo);
        uint32_t a0[4], a1[4];
        i8x4_to_f16x2(wa.x, a0[0], a0[2]);
        i8x4_to_f16x2(wb.x, a0[1], a0[3]);
        i8x4_to_f16x2(wa.y, a1[0], a1[2]);
        i8x4_to_f16x2(wb.y, a1[1], a1[3]);
        float sa, sbv;
        if constexpr (EXACT) {
            sa = ue8m0_to_f32((e0w >> (8 * b)) & 0xFF);
            sbv = ue8m0_to_f32((e1w >> (8 * b)) & 0xFF);
        } else {
            sa = b == 0 ? scale_fast<0>(e0w) : b == 1 ? scale_fast<1>(e0w)
                                             : b == 2 ? scale_fast<2>(e0w) : scale_fast<3>(e0w);
            sbv = b == 0 ? scale_fast<0>(e1w) : b == 1 ? scale_fast<1>(e1w)
                                              : b == 2 ? scale_fast<2>(e1w) : scale_fast<3>(e1w);
        }
#pragma unroll
        for (int h = 0; h < NH; ++h) {
            uint4 xv = xa;
            if (h == 1) xv = *reinterpret_cast<const uint4 *>(xhalf + (g + 8) * 128 + xo);
            const float z[4] = {0.f, 0.f, 0.f, 0.f};
            float p[4], q[4];
            mma_16816(p, a0, xv.x, xv.y, z);
            mma_16816(q, a1, xv.z, xv.w, p);
            acc[h][0] = fmaf(sa, q[0], acc[h][0]);
            acc[h][1] = fmaf(sa, q[1], acc[h][1]);
            acc[h][2] = fmaf(sbv, q[2], acc[h][2]);
            acc[h][3] = fmaf(sbv, q[3], acc[h][3]);
        }
    }
}

// NH = number of 8-column activation halves (1 for M <= 8, 2 for M <= 16).
template <int NH>
__global__ void __launch_bounds__(THREADS)
w8_gemv_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
               int M, const uint8_t *__restrict__ SW, int64_t ldsw, int sw_vec,
               __half *__restrict__ Y, int64_t ldy, int N, int K, int epi, unsigned *err,
               uint64_t timeout_ns) {
    using G = GCfg<NH>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto full_bar = [&](int s) { return sb + G::OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sb + G::OFF_BAR + 8u * (STAGES + s); };

    const int nrb = (N + ROWS - 1) / ROWS;     // 64-row blocks
    const int nkc = (K + KC - 1) / KC;         // 128-wide K chunks
    const int nblk = K / 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), CONSUMERS);
        }
        fence_barrier_init();
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
    }
    __syncthreads();

    if (warp == CONSUMERS) {
        // ------------------------------------------------------------------- producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            int issued = 0;
            bool ok = true;
            for (int rb = blockIdx.x; rb < nrb && ok; rb += gridDim.x) {
                for (int kc = 0; kc < nkc; ++kc) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1, timeout_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = sb + stage * G::STAGE;
                    mbar_arrive_expect_tx(full_bar(stage), G::STAGE);
                    tma_load_2d(st, &tmW, full_bar(stage), kc * KC, rb * ROWS);
                    tma_load_2d(st + G::W_BYTES, &tmX, full_bar(stage), kc * KC, 0);
                    tma_load_2d(st + G::W_BYTES + G::X_HALF, &tmX, full_bar(stage), kc * KC + 64, 0);
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok) atomicOr(err, ERR_PRODUCER);
            for (int i = max(0, issued - STAGES); i < issued; ++i)
                if (!mbar_wait(full_bar(i % STAGES), (i / STAGES) & 1, timeout_ns)) {
                    atomicOr(err, ERR_DRAIN);
                    break;
                }
        }
        return;
    }

    // ---------------------------------------------------------------------- consumers
    const int g = lane >> 2;    // fragment row group / activation row
    const int t = lane & 3;     // quad position: k offset 8 t inside a block
    const int r0 = warp * 16 + g;              // weight rows r0 and r0 + 8 of the 64-row tile
    const uint32_t sw = static_cast<uint32_t>(r0 & 7);   // 128-byte swizzle phase (same for r0+8)
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    for (int rb = blockIdx.x; rb < nrb && ok; rb += gridDim.x) {
        const int n0 = rb * ROWS + r0;
        const uint8_t *srow0 = SW + static_cast<int64_t>(min(n0, N - 1)) * ldsw;
        const uint8_t *srow1 = SW + static_cast<int64_t>(min(n0 + 8, N - 1)) * ldsw;
        float acc[NH][4];
#pragma unroll
        for (int h = 0; h < NH; ++h)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[h][i] = 0.f;
        // scale words for chunks kc .. kc + SCALE_AHEAD - 1, rotated each chunk
        uint32_t s0[SCALE_AHEAD], s1[SCALE_AHEAD];
#pragma unroll
        for (int i = 0; i < SCALE_AHEAD; ++i) {
            s0[i] = i < nkc ? scale_word(srow0, i, nblk, sw_vec) : 0x7F7F7F7Fu;
            s1[i] = i < nkc ? scale_word(srow1, i, nblk, sw_vec) : 0x7F7F7F7Fu;
        }
        for (int kc = 0; kc < nkc; ++kc) {
            const uint32_t e0w = s0[0], e1w = s1[0];
#pragma unroll
            for (int i = 0; i + 1 < SCALE_AHEAD; ++i) {
                s0[i] = s0[i + 1];
                s1[i] = s1[i + 1];
            }
            const int nxt = kc + SCALE_AHEAD;
            s0[SCALE_AHEAD - 1] = nxt < nkc ? scale_word(srow0, nxt, nblk, sw_vec) : 0x7F7F7F7Fu;
            s1[SCALE_AHEAD - 1] = nxt < nkc ? scale_word(srow1, nxt, nblk, sw_vec) : 0x7F7F7F7Fu;

            if (!mbar_wait(full_bar(stage), phase, timeout_ns)) {
                ok = false;
                break;
            }
            const uint8_t *st = smem + stage * G::STAGE;   // plain shared loads, schedulable
            const uint8_t *xs = st + G::W_BYTES;
            // Scale words of this stage: the fast decode builds 2^(e-127) by shifting the byte into
            // the fp32 exponent field; codes 0x00 (subnormal 2^-127) and 0xFF (NaN) take the exact
            // decode, chosen for the whole warp so the branch stays uniform.
            const bool exact = __any_sync(0xffffffffu, has_special_byte(e0w) || has_special_byte(e1w));
            if (exact)
                consume_stage<NH, true>(acc, st, xs, r0, sw, g, t, e0w, e1w);
            else
                consume_stage<NH, false>(acc, st, xs, r0, sw, g, t, e0w, e1w);
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(stage));
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1;
            }
        }
        if (!ok) break;
        // D fragment: acc[h][0..1] -> row n0, activations 8h + 2t (+1); acc[h][2..3] -> n0 + 8
#pragma unroll
        for (int h = 0; h < NH; ++h) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int m = 8 * h + 2 * t + (i & 1);
                const int n = n0 + ((i & 2) ? 8 : 0);
                if (m < M && n < N) {
                    __half *dst = Y + static_cast<int64_t>(m) * ldy + n;
                    float x = acc[h][i];
                    if (epi & EPI_ACC_BIT) x += __half2float(*dst);   // Y = relu?(X W^T + Y_old)
                    if (epi & EPI_RELU_BIT) x = fmaxf(x, 0.0f);
                    *dst = __float2half_rn(x);
                }
            }
        }
    }
    if (!ok && lane == 0) atomicOr(err, ERR_EPILOGUE);
}

template <int NH>
cudaError_t launch_nh(const __half *X, int64_t ldx, int M, const qgemm_tensor *W, __half *Y,
                      int64_t ldy, const qgi::LaunchCtx &ctx, bool *encode_ok) {
    using G = GCfg<NH>;
    const int N = static_cast<int>(W->rows), K = static_cast<int>(W->k);
    CUtensorMap tmW, tmX;
    *encode_ok = qgi::encode_tma_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, W->data, K, N, W->ld, KC,
                                    ROWS, CU_TENSOR_MAP_SWIZZLE_128B) &&
                 qgi::encode_tma_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, X, K, M, ldx * 2, 64,
                                    8 * NH, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!*encode_ok) return cudaErrorInvalidValue;
    auto kern = w8_gemv_kernel<NH>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
    if (e != cudaSuccess) return e;
    const int nrb = (N + ROWS - 1) / ROWS;
    const int per_sm = 232448 / G::SMEM;       // CTAs that fit in one SM's shared memory
    int grid = ctx.num_sms * (per_sm < 1 ? 1 : per_sm);
    if (grid > nrb) grid = nrb;
    const int sw_vec = (reinterpret_cast<uintptr_t>(W->scales) % 4 == 0 && W->lds % 4 == 0) ? 1 : 0;
    kern<<<grid, THREADS, G::SMEM, ctx.stream>>>(tmW, tmX, M, W->scales, W->lds, sw_vec, Y, ldy, N,
                                                 K, ctx.epi, ctx.err, ctx.timeout_ns);
    return cudaGetLastError();
}

}  // namespace

namespace qgi {

cudaError_t launch_w8_gemv(const __half *X, int64_t ldx, int M, const qgemm_tensor *W,
                           __half *Y, int64_t ldy, const LaunchCtx &ctx, bool *encode_ok) {
    if (M <= 8) return launch_nh<1>(X, ldx, M, W, Y, ldy, ctx, encode_ok);
    return launch_nh<2>(X, ldx, M, W, Y, ldy, ctx, encode_ok);
}

}  // namespace qgi
