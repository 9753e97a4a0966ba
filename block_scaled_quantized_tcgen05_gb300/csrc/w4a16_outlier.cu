// w4a16_outlier.cu -- exact recomputation of the outlier rows of a weight-only int4 GEMM.
//
// The int4 GEMMs fold each UE8M0 block scale into the fp16 weight, q * 2^(e-127), which is
// exact only for scale bytes 103..139 (w4a16_convert.cuh).  The product the library defines --
// "TensorOps: quantized matmul ..." (section "M2 = block-32 fp16 scaling": each 32-block of
// weights times its block's scale, then the product with the activations; section
// "Kernel-phase findings": the scale is an E8M0 power of two) -- holds for every scale byte.
// A weight row with a nonzero weight in a block whose byte lies outside that window (and is not
// the NaN code 255) is an outlier row; the GEMM kernels write such a column with the
// out-of-window blocks as zero (or, when accumulating, leave it alone), and this kernel, run
// right after them on the same stream, writes it again from the definition:
//
//   C[m, n] = fp16_rn( relu?( sum_b 2^(e_b - 127) * P_b[m] [+ C_old[m, n]] ) ),
//   P_b[m]  = sum over the 32 k of block b of A[m, k] * q[n, k]   (fp32; each product is exact)
//
// with the block partials scaled and summed in fp64 (every 2^(e-127) and every fp32 partial
// times it is a double, so nothing over- or underflows before the single fp16 rounding).
//
// Grid: x over 256-row groups of W (one thread tests one row), y over token groups of A (as
// many as fit beside x in one CTA per SM).  Each CTA marks its group's outlier rows in a 256-bit
// mask in shared memory and, for each in row order, has its eight warps take the tokens of its
// token group in turn: lane l
// reads the 16-byte chunks l, l + 32, ... of the token's activation row (8 k each, four chunks
// per block), the four lanes of a block add their partials in a fixed order, and the fp64 block
// terms are added by a fixed shuffle tree, so the result does not depend on timing.
//
// The kernel is launched with programmatic stream serialization and the GEMM kernels release it
// at their start (griddepcontrol.launch_dependents), so its CTAs take the SM room the GEMM leaves
// (about 10 K registers and 1.8 KB of shared memory per SM) and read the scale plane while the GEMM
// runs.  Every thread then waits for the GEMM to complete (griddepcontrol.wait) before touching
// C -- and before exiting, so that this grid's completion, which later work on the stream waits
// for, implies the GEMM's.  With no outlier row (the usual case) that wait is all that is left.
#include <cuda_fp16.h>

#include "qgemm_common.cuh"
#include "qgemm_internal.h"
#include "qgemm_ptx.cuh"
#include "w4a16_convert.cuh"

namespace {

using namespace qg;

constexpr int OT_ROWS = 256;     // weight rows tested per CTA (one per thread)
constexpr int OT_MIN_TOKENS = 64;   // smallest token group worth a CTA of its own
constexpr int OT_THREADS = 256;
constexpr int OT_WARPS = OT_THREADS / 32;

// 2^(e - 127) as a double; NaN for 255.
__device__ __forceinline__ double ue8m0_f64(uint32_t e) {
    if (e == UE8M0_NAN) return __longlong_as_double(0x7FF8000000000000LL);
    return __longlong_as_double(static_cast<long long>(e + (1023u - 127u)) << 52);
}

__device__ __forceinline__ uint16_t f64_to_f16_rn(double x) {
    uint16_t h;
    asm("cvt.rn.f16.f64 %0, %1;" : "=h"(h) : "d"(x));
    return h;
}

// Signed int4 nibble j (0..7) of a packed word, as a float.
__device__ __forceinline__ float nibble_f(uint32_t w, int j) {
    return static_cast<float>(static_cast<int>(w << (28 - 4 * j)) >> 28);
}

__global__ void __launch_bounds__(OT_THREADS, 6)   // <= 40 registers: fits beside the GEMMs
w4a16_outlier_kernel(const __half *__restrict__ A, int64_t lda, int M,
                     const uint8_t *__restrict__ W, int64_t ldw, const uint8_t *__restrict__ S,
                     int64_t lds, int N, int K, __half *__restrict__ C, int64_t ldc, int epi,
                     int tokens_per_cta) {
    __shared__ uint32_t mask[OT_ROWS / 32];   // bit t of word w: row 32 w + t of the group
    const int t = static_cast<int>(threadIdx.x);
    const int warp = t >> 5, lane = t & 31;
    const int n = static_cast<int>(blockIdx.x) * OT_ROWS + t;
    const bool mine = n < N && w4_row_is_outlier(S + static_cast<int64_t>(n) * lds,
                                                 W + static_cast<int64_t>(n) * ldw, K / 32);
    const uint32_t bits = __ballot_sync(0xFFFFFFFFu, mine);
    if (lane == 0) mask[warp] = bits;
    __syncthreads();
    uint32_t any = 0;
#pragma unroll
    for (int w = 0; w < OT_ROWS / 32; ++w) any |= mask[w];
    griddep_wait();   // the GEMM has written C (see the file comment)
    if (any == 0) return;

    const int nchunk = K / 8;   // 16-byte activation chunks per token row (a multiple of 4)
    for (int r = 0; r < OT_ROWS; ++r) {
        if (!((mask[r >> 5] >> (r & 31)) & 1u)) continue;
        const int nn = static_cast<int>(blockIdx.x) * OT_ROWS + r;
        const uint8_t *wrow = W + static_cast<int64_t>(nn) * ldw;
        const uint8_t *srow = S + static_cast<int64_t>(nn) * lds;
        for (int64_t m0 = static_cast<int64_t>(blockIdx.y) * tokens_per_cta; m0 < M;
             m0 += static_cast<int64_t>(gridDim.y) * tokens_per_cta) {
            const int m_end = static_cast<int>(m0 + tokens_per_cta < M ? m0 + tokens_per_cta : M);
            for (int m = static_cast<int>(m0) + warp; m < m_end; m += OT_WARPS) {
                const __half *arow = A + static_cast<int64_t>(m) * lda;
                double acc = 0.0;
                for (int c0 = 0; c0 < nchunk; c0 += 32) {
                    const int c = c0 + lane;
                    float p = 0.0f;
                    uint32_t e = 127u;
                    if (c < nchunk) {
                        const uint4 av = __ldg(reinterpret_cast<const uint4 *>(arow) + c);
                        const uint32_t wv = __ldg(reinterpret_cast<const uint32_t *>(wrow) + c);
                        const uint32_t aw[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const __half2 h = *reinterpret_cast<const __half2 *>(&aw[j]);
                            p = fmaf(__low2float(h), nibble_f(wv, 2 * j), p);
                            p = fmaf(__high2float(h), nibble_f(wv, 2 * j + 1), p);
                        }
                        e = __ldg(srow + (c >> 2));
                    }
                    // the block's four chunks (lanes 4g .. 4g + 3), in a fixed order
                    p += __shfl_xor_sync(0xFFFFFFFFu, p, 1);
                    p += __shfl_xor_sync(0xFFFFFFFFu, p, 2);
                    if (c < nchunk && (lane & 3) == 0)
                        acc += static_cast<double>(p) * ue8m0_f64(e);
                }
                acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 4);
                acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 8);
                acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 16);
                if (lane == 0) {
                    __half *dst = C + static_cast<int64_t>(m) * ldc + nn;
                    double x = acc;
                    if (epi & EPI_ACC_BIT) x += static_cast<double>(__half2float(*dst));
                    if (epi & EPI_RELU_BIT) x = x > 0.0 ? x : 0.0;   // NaN -> +0, as fmaxf
                    *reinterpret_cast<uint16_t *>(dst) = f64_to_f16_rn(x);
                }
            }
        }
    }
}

}  // namespace

namespace qgi {

cudaError_t launch_w4a16_outliers(const __half *A, int64_t lda, int M, const qgemm_tensor *W,
                                  __half *C, int64_t ldc, const LaunchCtx &ctx) {
    const int N = static_cast<int>(W->rows), K = static_cast<int>(W->k);
    const int gx = (N + OT_ROWS - 1) / OT_ROWS;
    // token groups: as many as fit one CTA per SM beside the row groups, at least 64 tokens each
    int gy = ctx.num_sms / gx;
    const int max_gy = (M + OT_MIN_TOKENS - 1) / OT_MIN_TOKENS;
    if (gy > max_gy) gy = max_gy;
    if (gy > 65535) gy = 65535;
    if (gy < 1) gy = 1;
    const int tokens = static_cast<int>((static_cast<int64_t>(M) + gy - 1) / gy);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(gx, gy);
    cfg.blockDim = dim3(OT_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, w4a16_outlier_kernel, A, lda, M, W->data, W->ld, W->scales,
                              W->lds, N, K, C, ldc, ctx.epi, tokens);
}

}  // namespace qgi
