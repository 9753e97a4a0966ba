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
// consumers' fragment reads from shared memory are free of bank conflicts.  Work is split along K
// inside a stage: consumer warp w takes 32-block w of every stage for all 64 rows, as four 16-row
// MMA fragments that share one activation fragment (each activation byte is read from shared
// memory once per stage instead of once per row fragment).  Per fragment a lane quad (t = 0..3)
// takes 8 consecutive int8 of rows g and g+8, converts them exactly to fp16 with a byte-permute
// into the mantissa of 1024 (a published integer-to-half technique), and feeds two k16 MMAs; the
// 32 k of a block are permuted identically for weights and activations, so the dot product is
// unchanged.  The block's fp32 partial sum is scaled by 2^(e-127) (exact) and added to the warp's
// running fp32 sum, so every UE8M0 scale is handled exactly.  At the end of a row block the four
// warps' sums are added in a fixed order (warp 0, 1, 2, 3) through shared memory, so results do
// not depend on timing.  CTAs are persistent over 64-row blocks.
#include <cuda_fp16.h>

#include "qgemm_common.cuh"
#include "qgemm_debug.cuh"
#include "qgemm_internal.h"
#include "qgemm_ptx.cuh"

namespace {

using namespace qg;

constexpr int CONSUMERS = 4;
constexpr int THREADS = (CONSUMERS + 1) * 32;
constexpr int KC = 128;                     // K per stage (bytes of int8) = four 32-blocks

// NH: 8-column activation halves (1: M <= 8, 2: M <= 16); NF: 16-row weight fragments per CTA
// (a row block is 16 NF rows).  M <= 8 takes 48-row blocks with six stages: 598 CTAs at
// N = 28672, four per SM (16 consumer warps to hide the latency of the loads, conversions and
// MMAs; with 64-row blocks only three fit and 448 row blocks fill 2.95 per SM).
template <int NH, int NF, int STAGES_>
struct GCfg {
    static constexpr int STAGES = STAGES_;
    static constexpr int ROWS = 16 * NF;
    static constexpr uint32_t W_BYTES = ROWS * KC;            // 6 or 8 KB
    static constexpr uint32_t X_HALF = 8 * NH * 128;          // one 64-wide half of the X slice
    static constexpr uint32_t X_BYTES = 2 * X_HALF;
    static constexpr uint32_t STAGE = W_BYTES + X_BYTES;
    static constexpr uint32_t OFF_BAR = STAGES * STAGE;       // full[S], empty[S]
    static constexpr uint32_t OFF_RBAR = OFF_BAR + 2 * STAGES * 8;   // reduction full, empty
    static constexpr uint32_t OFF_RED = OFF_RBAR + 16;
    // partial sums handed between warps, one activation half at a time: [warp][NF][4][lane]
    static constexpr uint32_t RED_BYTES = CONSUMERS * NF * 4 * 32 * 4;
    static constexpr uint32_t SMEM = OFF_RED + RED_BYTES + 1024;
    static_assert(STAGE % 1024 == 0, "stages stay 1 KB aligned for the 128-byte swizzle");
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
// independent fragments.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1, const float (&c)[4]) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
          "f"(c[2]), "f"(c[3]));
}

// Scale bytes of blocks 16 G .. 16 G + 15 of one row (the four 32-blocks of four consecutive
// stages) as four little-endian words; bytes past the row's last block read as 127 (2^0; their
// data is zero-filled).  vec: 2 = the row is 16-byte aligned, 1 = 4-byte aligned, 0 = bytes.
__device__ __forceinline__ uint4 scale_group(const uint8_t *row, int G, int nblk, int vec) {
    const int b0 = 16 * G;
    if (vec == 2 && b0 + 16 <= nblk) return __ldg(reinterpret_cast<const uint4 *>(row + b0));
    uint32_t v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int bj = b0 + 4 * j;
        if (vec >= 1 && bj + 4 <= nblk) {
            v[j] = __ldg(reinterpret_cast<const uint32_t *>(row + bj));
        } else {
            uint32_t x = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                x |= static_cast<uint32_t>(bj + i < nblk ? __ldg(row + bj + i) : 127) << (8 * i);
            v[j] = x;
        }
    }
    return make_uint4(v[0], v[1], v[2], v[3]);
}

// True if some byte of w is 0x00 or 0xFF (the scale codes the shift decode does not cover).
__device__ __forceinline__ bool has_special_byte(uint32_t w) {
    const uint32_t z = (w - 0x01010101u) & ~w & 0x80808080u;     // a zero byte
    const uint32_t n = ~w;
    const uint32_t f = (n - 0x01010101u) & ~n & 0x80808080u;     // a 0xFF byte
    return (z | f) != 0u;
}

// The products of one stage: this warp's 32-block for all 64 rows, accumulated into acc with the
// stage's block scales (byte sh / 8 of e0[f], e1[f]).  Plain shared loads and pure MMAs, so two calls
// in a row can be interleaved by the compiler.
template <int NH, int NF, bool EXACT>
__device__ __forceinline__ void stage_math(float (&acc)[NF][NH][4], const uint8_t *st, uint32_t wrow,
                                           uint32_t xoff, const uint32_t (&e0)[NF],
                                           const uint32_t (&e1)[NF], uint32_t sh) {
    const uint8_t *xs = st + 16 * NF * KC;
    const uint4 xa = *reinterpret_cast<const uint4 *>(xs + xoff);
    uint4 xb = xa;
    if constexpr (NH == 2) xb = *reinterpret_cast<const uint4 *>(xs + xoff + 8 * 128);
#pragma unroll
    for (int f = 0; f < NF; ++f) {
        const uint2 wa = *reinterpret_cast<const uint2 *>(st + wrow + f * 16 * 128);
        const uint2 wb = *reinterpret_cast<const uint2 *>(st + wrow + (f * 16 + 8) * 128);
        uint32_t a0[4], a1[4];
        i8x4_to_f16x2(wa.x, a0[0], a0[2]);
        i8x4_to_f16x2(wb.x, a0[1], a0[3]);
        i8x4_to_f16x2(wa.y, a1[0], a1[2]);
        i8x4_to_f16x2(wb.y, a1[1], a1[3]);
        const uint32_t b0 = (e0[f] >> sh) & 0xFFu, b1 = (e1[f] >> sh) & 0xFFu;
        const float sa = EXACT ? ue8m0_to_f32(b0) : __uint_as_float(b0 << 23);
        const float sbv = EXACT ? ue8m0_to_f32(b1) : __uint_as_float(b1 << 23);
#pragma unroll
        for (int h = 0; h < NH; ++h) {
            const uint4 xv = h == 0 ? xa : xb;
            const float z[4] = {0.f, 0.f, 0.f, 0.f};
            float p[4], q[4];
            mma_16816(p, a0, xv.x, xv.y, z);
            mma_16816(q, a1, xv.z, xv.w, p);
            acc[f][h][0] = fmaf(sa, q[0], acc[f][h][0]);
            acc[f][h][1] = fmaf(sa, q[1], acc[f][h][1]);
            acc[f][h][2] = fmaf(sbv, q[2], acc[f][h][2]);
            acc[f][h][3] = fmaf(sbv, q[3], acc[f][h][3]);
        }
    }
}

// Up to four stages of one scale group (stages 4 G0 .. 4 G0 + 3 that exist), taken two at a time:
// both are waited for, their products formed together (twice the independent work between the
// warp's waits), added to acc in stage order, and both handed back.  e0[f] / e1[f] hold the scale
// bytes of rows 16 f + g / 16 f + g + 8 for this warp's block of each stage (stage j in byte j).
// EXACT selects the decode for the whole group: the shift decode builds 2^(e-127) by moving the
// byte into the fp32 exponent field; codes 0x00 (subnormal 2^-127) and 0xFF (NaN) need the exact one.
template <int NH, int NF, bool EXACT, int STAGES>
__device__ __forceinline__ bool run_group(float (&acc)[NF][NH][4], const uint8_t *smem, uint32_t sb,
                                          uint32_t stage_bytes, uint32_t off_bar, int nst,
                                          uint32_t wrow, uint32_t xoff, const uint32_t (&e0)[NF],
                                          const uint32_t (&e1)[NF], uint32_t &stage, uint32_t &phase,
                                          int lane, uint64_t timeout_ns) {
#pragma unroll
    for (int j = 0; j < 4; j += 2) {
        if (j >= nst) break;
        const bool two = j + 1 < nst;
        uint32_t stage2 = stage + 1, phase2 = phase;
        if (stage2 == STAGES) {
            stage2 = 0;
            phase2 ^= 1;
        }
        const uint32_t full = sb + off_bar + 8u * stage, full2 = sb + off_bar + 8u * stage2;
        if (!mbar_wait(full, phase, timeout_ns)) return false;
        if (two && !mbar_wait(full2, phase2, timeout_ns)) return false;
        // Reconverge before the warp-wide mma.sync.aligned: lane 0 alone took the arrive branch of the
        // previous stages and every lane polls the barriers on its own.
        __syncwarp();
        stage_math<NH, NF, EXACT>(acc, smem + stage * stage_bytes, wrow, xoff, e0, e1, 8u * j);
        if (two)
            stage_math<NH, NF, EXACT>(acc, smem + stage2 * stage_bytes, wrow, xoff, e0, e1,
                                      8u * (j + 1));
        // Hand the stages back.  Their operands were read through the generic proxy and the producer's
        // next TMA writes them through the async proxy: each lane orders its reads before that write
        // with a proxy fence (measured on this GPU: without it, whole 64-row blocks picked up data of
        // the next fill now and then).
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(full + 8u * STAGES);
            if (two) mbar_arrive(full2 + 8u * STAGES);
        }
        stage = two ? (stage2 + 1 == STAGES ? 0 : stage2 + 1) : stage2;
        phase = two ? (stage2 + 1 == STAGES ? phase2 ^ 1 : phase2) : phase2;
    }
    return true;
}

// NH = number of 8-column activation halves (1 for M <= 8, 2 for M <= 16); NF, STAGES as GCfg.
template <int NH, int NF, int STAGES_>
__global__ void __launch_bounds__(THREADS)
w8_gemv_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
               int M, const uint8_t *__restrict__ SW, int64_t ldsw, int sw_vec,
               __half *__restrict__ Y, int64_t ldy, int N, int K, int epi, unsigned *err,
               uint64_t timeout_ns) {
    using G = GCfg<NH, NF, STAGES_>;
    constexpr int STAGES = G::STAGES;
    constexpr int ROWS = G::ROWS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    griddep_launch_dependents();   // a dependent launch (e.g. a clock probe) may run beside
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto full_bar = [&](int s) { return sb + G::OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sb + G::OFF_BAR + 8u * (STAGES + s); };
    const uint32_t red_full = sb + G::OFF_RBAR, red_empty = sb + G::OFF_RBAR + 8;
    float *red = reinterpret_cast<float *>(smem + G::OFF_RED);

    const int nrb = (N + ROWS - 1) / ROWS;     // row blocks
    const int nkc = (K + KC - 1) / KC;         // 128-wide K chunks (stages)
    const int ngrp = (nkc + 3) / 4;            // groups of four stages (one 16-byte scale load)
    const int nblk = K / 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), CONSUMERS);
        }
        mbar_init(red_full, 32 * CONSUMERS);
        mbar_init(red_empty, 32 * CONSUMERS);
        fence_barrier_init();
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
    }
    __syncthreads();
    // Launched as a programmatic dependent: the CTAs may be resident before the kernel ahead of
    // this one on the stream has finished.  Nothing in memory is touched before it has.
    griddep_wait();

    if (warp == CONSUMERS) {
        // ------------------------------------------------------------------- producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            int issued = 0;
            bool ok = true;
            // The weights are read once: evict-first lines in L2, so the stream replaces its own
            // lines instead of pushing out (and writing back) what earlier kernels left there.
            const uint64_t stream_once = l2_policy_evict_first();
            for (int rb = blockIdx.x; rb < nrb && ok; rb += gridDim.x) {
                for (int kc = 0; kc < nkc; ++kc) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1, timeout_ns)) {
                        ok = false;
                        break;
                    }
                    // debug build: innermost coordinates multiples of 16 bytes, the row block
                    // inside N
                    if (!QG_IN_BOUNDS(err, (kc * KC) % 16 == 0 && rb * ROWS < N)) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = sb + stage * G::STAGE;
                    mbar_arrive_expect_tx(full_bar(stage), G::STAGE);
                    tma_load_2d_hint(st, &tmW, full_bar(stage), kc * KC, rb * ROWS, stream_once);
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
    const int w = warp;         // the 32-block of every stage this warp takes
    const int g = lane >> 2;    // fragment row group / activation row
    const int t = lane & 3;     // quad position: k offset 8 t inside the block
    // weights: bytes 32 w + 8 t .. +8 of rows 16 f + g and 16 f + g + 8 (swizzle phase g for all)
    const uint32_t wrow = static_cast<uint32_t>(g) * 128 +
                          ((static_cast<uint32_t>(2 * w + (t >> 1)) ^ static_cast<uint32_t>(g)) << 4) +
                          static_cast<uint32_t>((t & 1) * 8);
    // activations: halves 32 w + 8 t .. +8 of X row g (row g + 8 is 1 KB further on)
    const uint32_t xoff = static_cast<uint32_t>(w >> 1) * G::X_HALF + static_cast<uint32_t>(g) * 128 +
                          ((static_cast<uint32_t>(4 * (w & 1) + t) ^ static_cast<uint32_t>(g)) << 4);
    // byte w of two scale words (a 16-byte scale group holds block w of stage j in byte 4 j + w)
    const uint32_t sel = static_cast<uint32_t>(w) | (static_cast<uint32_t>(4 + w) << 4);
    uint32_t stage = 0, phase = 0, rphase = 0;
    bool ok = true;
    for (int rb = blockIdx.x; rb < nrb && ok; rb += gridDim.x) {
        // this lane loads the scale rows of fragment t (rows 16 t + g and 16 t + g + 8) and shares
        // them with the other lanes of its quad (t >= NF: no fragment, neutral bytes)
        const bool has_frag = t < NF;
        const int nA = rb * ROWS + 16 * t + g;
        const uint8_t *srowA = SW + static_cast<int64_t>(min(nA, N - 1)) * ldsw;
        const uint8_t *srowB = SW + static_cast<int64_t>(min(nA + 8, N - 1)) * ldsw;
        float acc[NF][NH][4];
#pragma unroll
        for (int f = 0; f < NF; ++f)
#pragma unroll
            for (int h = 0; h < NH; ++h)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[f][h][i] = 0.f;
        const uint4 neutral = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
        uint4 rawA = has_frag ? scale_group(srowA, 0, nblk, sw_vec) : neutral;
        uint4 rawB = has_frag ? scale_group(srowB, 0, nblk, sw_vec) : neutral;
        for (int G0 = 0; G0 < ngrp && ok; ++G0) {
            const uint4 cA = rawA, cB = rawB;
            if (G0 + 1 < ngrp && has_frag) {        // one group ahead
                rawA = scale_group(srowA, G0 + 1, nblk, sw_vec);
                rawB = scale_group(srowB, G0 + 1, nblk, sw_vec);
            }
            // this warp's block of each of the group's four stages, stage j in byte j
            const uint32_t pA = __byte_perm(__byte_perm(cA.x, cA.y, sel), __byte_perm(cA.z, cA.w, sel),
                                            0x5410u);
            const uint32_t pB = __byte_perm(__byte_perm(cB.x, cB.y, sel), __byte_perm(cB.z, cB.w, sel),
                                            0x5410u);
            // the lanes together hold every row of the block: one vote decides the decode
            const bool exact = __any_sync(0xffffffffu, has_special_byte(pA) || has_special_byte(pB));
            uint32_t e0[NF], e1[NF];    // scale bytes of rows 16 f + g (e0) and 16 f + g + 8 (e1)
#pragma unroll
            for (int f = 0; f < NF; ++f) {
                e0[f] = __shfl_sync(0xffffffffu, pA, (g << 2) | f);
                e1[f] = __shfl_sync(0xffffffffu, pB, (g << 2) | f);
            }
            const int nst = min(4, nkc - 4 * G0);
            ok = exact ? run_group<NH, NF, true, STAGES>(acc, smem, sb, G::STAGE, G::OFF_BAR, nst,
                                                         wrow, xoff, e0, e1, stage, phase, lane,
                                                         timeout_ns)
                       : run_group<NH, NF, false, STAGES>(acc, smem, sb, G::STAGE, G::OFF_BAR, nst,
                                                          wrow, xoff, e0, e1, stage, phase, lane,
                                                          timeout_ns);
        }
        if (!ok) break;
        // Row block done: warp w < NF finishes fragment w.  Every warp hands its sums over through
        // shared memory, one activation half at a time; the four partial sums of a fragment are
        // added in warp order.  Waits are bounded like the stage waits.
#pragma unroll
        for (int h = 0; h < NH; ++h) {
            if (!mbar_wait(red_empty, rphase ^ 1, timeout_ns)) {
                ok = false;
                break;
            }
#pragma unroll
            for (int f = 0; f < NF; ++f) {
                if (f == w) continue;
#pragma unroll
                for (int i = 0; i < 4; ++i) red[((w * NF + f) * 4 + i) * 32 + lane] = acc[f][h][i];
            }
            mbar_arrive(red_full);
            if (!mbar_wait(red_full, rphase, timeout_ns)) {
                ok = false;
                break;
            }
            float own[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int f = 0; f < NF; ++f)
                if (f == w)
#pragma unroll
                    for (int i = 0; i < 4; ++i) own[i] = acc[f][h][i];
            float sum[4] = {0.f, 0.f, 0.f, 0.f};
            if (w < NF) {
#pragma unroll
                for (int u = 0; u < CONSUMERS; ++u)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        sum[i] += u == w ? own[i] : red[((u * NF + w) * 4 + i) * 32 + lane];
            }
            mbar_arrive(red_empty);
            rphase ^= 1;
            if (w >= NF) continue;
            // D fragment: sum[0..1] -> row n0, activations 8h + 2t (+1); sum[2..3] -> n0 + 8
            const int n0 = rb * ROWS + 16 * w + g;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int m = 8 * h + 2 * t + (i & 1);
                const int n = n0 + ((i & 2) ? 8 : 0);
                if (m < M && n < N) {
                    __half *dst = Y + static_cast<int64_t>(m) * ldy + n;
                    float x = sum[i];
                    if (epi & EPI_ACC_BIT) x += __half2float(*dst);   // Y = relu?(X W^T + Y_old)
                    if (epi & EPI_RELU_BIT) x = fmaxf(x, 0.0f);
                    *dst = __float2half_rn(x);
                }
            }
        }
    }
    if (!ok && lane == 0) atomicOr(err, ERR_EPILOGUE);
}

template <int NH, int NF, int STAGES>
cudaError_t launch_nh(const __half *X, int64_t ldx, int M, const qgemm_tensor *W, __half *Y,
                      int64_t ldy, const qgi::LaunchCtx &ctx, bool *encode_ok) {
    using G = GCfg<NH, NF, STAGES>;
    constexpr int ROWS = G::ROWS;
    const int N = static_cast<int>(W->rows), K = static_cast<int>(W->k);
    CUtensorMap tmW, tmX;
    *encode_ok = qgi::encode_tma_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, W->data, K, N, W->ld, KC,
                                    ROWS, CU_TENSOR_MAP_SWIZZLE_128B) &&
                 qgi::encode_tma_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, X, K, M, ldx * 2, 64,
                                    8 * NH, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!*encode_ok) return cudaErrorInvalidValue;
    auto kern = w8_gemv_kernel<NH, NF, STAGES>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
    if (e != cudaSuccess) return e;
    const int nrb = (N + ROWS - 1) / ROWS;
    const int per_sm = 233472 / (G::SMEM + 1024);   // CTAs that fit in one SM's shared memory
    int grid = ctx.num_sms * (per_sm < 1 ? 1 : per_sm);
    if (grid > nrb) grid = nrb;
    const uintptr_t sp = reinterpret_cast<uintptr_t>(W->scales);
    const int sw_vec = (sp % 16 == 0 && W->lds % 16 == 0) ? 2 : (sp % 4 == 0 && W->lds % 4 == 0) ? 1 : 0;
    // A programmatic dependent of the kernel ahead on the stream: launch, set-up and barrier
    // initialisation overlap that kernel's last CTAs (each kernel boundary otherwise costs about
    // 3 us on this GPU, against a 38 us weight stream).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = G::SMEM;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmW, tmX, M, W->scales, W->lds, sw_vec, Y, ldy, N, K,
                              ctx.epi, ctx.err, ctx.timeout_ns);
}

}  // namespace

namespace qgi {

cudaError_t launch_w8_gemv(const __half *X, int64_t ldx, int M, const qgemm_tensor *W,
                           __half *Y, int64_t ldy, const LaunchCtx &ctx, bool *encode_ok) {
    if (M <= 8) return launch_nh<1, 3, 6>(X, ldx, M, W, Y, ldy, ctx, encode_ok);
    return launch_nh<2, 4, 5>(X, ldx, M, W, Y, ldy, ctx, encode_ok);
}

}  // namespace qgi
