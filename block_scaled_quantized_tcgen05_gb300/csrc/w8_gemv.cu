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
// Each warp owns 16 weight rows over all of K.  Per 32-element block a lane quad (t = 0..3) loads
// 8 consecutive int8 of rows g and g+8 (8-byte loads, one 32-byte sector per row per quad),
// converts them exactly to fp16 with a byte-permute into the mantissa of 1024 (a published
// integer-to-half technique), and feeds two k16 MMAs.  The 32 k of a block are permuted the same
// way for weights and activations, so the dot product is unchanged.  The block's fp32 partial
// sum is then scaled by 2^(e-127) (exact) and added to the running fp32 sum, so every UE8M0 scale
// is handled exactly.
#include <cuda_fp16.h>

#include "qgemm_internal.h"
#include "qgemm_ptx.cuh"

namespace {

using namespace qg;

constexpr int WARPS = 4;
constexpr int THREADS = WARPS * 32;
constexpr int ROWS_PER_WARP = 16;
constexpr int UNROLL = 8;  // blocks of 32 in flight per warp

// 4 int8 (one 32-bit word) -> two fp16x2 holding the exact integers (q0,q1), (q2,q3).
__device__ __forceinline__ void i8x4_to_f16x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;                  // q + 128, as unsigned bytes
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x5140u);  // halves 0x64|b0, 0x64|b1
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x5342u);  // halves 0x64|b2, 0x64|b3
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2 *>(&a), bias);  // (1024+u)-1152
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2 *>(&b), bias);
    lo = *reinterpret_cast<const uint32_t *>(&ha);
    hi = *reinterpret_cast<const uint32_t *>(&hb);
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1, const float (&c)[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
          "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ uint2 ld_stream_u2(const uint8_t *p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
                 : "=r"(v.x), "=r"(v.y)
                 : "l"(p));
    return v;
}

// NH = number of 8-column activation halves (1 for M <= 8, 2 for M <= 16).
template <int NH>
__global__ void __launch_bounds__(THREADS)
w8_gemv_kernel(const __half *__restrict__ X, int64_t ldx, int M, const uint8_t *__restrict__ W,
               int64_t ldw, const uint8_t *__restrict__ SW, int64_t ldsw, __half *__restrict__ Y,
               int64_t ldy, int N, int K) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;  // row group inside the 16-row tile / activation row
    const int t = lane & 3;   // quad position: k offset 8 t inside a block
    const int n0 = (blockIdx.x * WARPS + warp) * ROWS_PER_WARP;
    if (n0 >= N) return;
    const int r0 = min(n0 + g, N - 1);       // rows past N read row N-1 and are never stored
    const int r1 = min(n0 + g + 8, N - 1);
    const uint8_t *w0 = W + static_cast<int64_t>(r0) * ldw + 8 * t;
    const uint8_t *w1 = W + static_cast<int64_t>(r1) * ldw + 8 * t;
    const uint8_t *s0 = SW + static_cast<int64_t>(r0) * ldsw;
    const uint8_t *s1 = SW + static_cast<int64_t>(r1) * ldsw;
    // activation rows g (first half) and g + 8 (second half); rows >= M read as zero
    const __half *x0 = X + static_cast<int64_t>(min(g, M - 1)) * ldx + 8 * t;
    const __half *x1 = X + static_cast<int64_t>(min(g + 8, M - 1)) * ldx + 8 * t;
    const bool xv0 = g < M;
    const bool xv1 = (g + 8) < M;

    float acc[NH][4];
#pragma unroll
    for (int h = 0; h < NH; ++h)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[h][i] = 0.f;

    const int nblk = K / 32;
#pragma unroll 1
    for (int b0 = 0; b0 < nblk; b0 += UNROLL) {
        uint2 wa[UNROLL], wb[UNROLL];
        uint4 xa[UNROLL], xb[UNROLL];
        uint32_t ea[UNROLL], eb[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int b = b0 + u;
            if (b < nblk) {
                wa[u] = ld_stream_u2(w0 + 32 * b);
                wb[u] = ld_stream_u2(w1 + 32 * b);
                ea[u] = __ldg(s0 + b);
                eb[u] = __ldg(s1 + b);
                xa[u] = xv0 ? __ldg(reinterpret_cast<const uint4 *>(x0 + 32 * b))
                            : make_uint4(0, 0, 0, 0);
                if (NH > 1)
                    xb[u] = xv1 ? __ldg(reinterpret_cast<const uint4 *>(x1 + 32 * b))
                                : make_uint4(0, 0, 0, 0);
            } else {
                wa[u] = wb[u] = make_uint2(0, 0);
                ea[u] = eb[u] = 127;
                xa[u] = xb[u] = make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            // step 0 uses bytes 0..3 of each row's 8, step 1 bytes 4..7
            uint32_t a0[4], a1[4];
            i8x4_to_f16x2(wa[u].x, a0[0], a0[2]);
            i8x4_to_f16x2(wb[u].x, a0[1], a0[3]);
            i8x4_to_f16x2(wa[u].y, a1[0], a1[2]);
            i8x4_to_f16x2(wb[u].y, a1[1], a1[3]);
            const float sa = ue8m0_to_f32(ea[u]);
            const float sbv = ue8m0_to_f32(eb[u]);
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                const uint4 xv = (h == 0) ? xa[u] : xb[u];
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

    // D fragment: acc[h][0..1] -> rows n0+g, activations 8h + 2t, 8h + 2t + 1;
    //             acc[h][2..3] -> rows n0+g+8, same activations.
#pragma unroll
    for (int h = 0; h < NH; ++h) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = 8 * h + 2 * t + (i & 1);
            const int n = n0 + g + ((i & 2) ? 8 : 0);
            if (m < M && n < N) Y[static_cast<int64_t>(m) * ldy + n] = __float2half_rn(acc[h][i]);
        }
    }
}

}  // namespace

namespace qgi {

cudaError_t launch_w8_gemv(const __half *X, int64_t ldx, int M, const qgemm_tensor *W,
                           __half *Y, int64_t ldy, const LaunchCtx &ctx) {
    const int N = static_cast<int>(W->rows), K = static_cast<int>(W->k);
    const int rows_per_cta = WARPS * ROWS_PER_WARP;
    const int grid = (N + rows_per_cta - 1) / rows_per_cta;
    if (M <= 8)
        w8_gemv_kernel<1><<<grid, THREADS, 0, ctx.stream>>>(X, ldx, M, W->data, W->ld, W->scales,
                                                            W->lds, Y, ldy, N, K);
    else
        w8_gemv_kernel<2><<<grid, THREADS, 0, ctx.stream>>>(X, ldx, M, W->data, W->ld, W->scales,
                                                            W->lds, Y, ldy, N, K);
    return cudaGetLastError();
}

}  // namespace qgi
