// splitk_reduce.cu -- the second half of a split-K GEMM: fp32 partial planes -> fp16 C.
//
// A GEMM whose output has too few tiles to occupy the GPU (at most 128 rows on one side: a
// decode-sized batch against a weight matrix) cuts the sum over K into `splits` consecutive
// k ranges, one CTA per (tile, range), and each CTA writes its unrounded fp32 sum into plane s of
// a scratch buffer P (M rows of ldp floats per plane, 16-byte aligned rows).  This kernel adds the
// planes in split order, s = 0, 1, ..., splits - 1, so the result does not depend on which CTA
// finished first, applies the fused epilogue (C_old added when accumulating, then ReLU) and rounds
// once to fp16, as the one-pass epilogue does.
//
// Each thread takes four consecutive columns of one row (16-byte loads from every plane; the
// planes sit in L2, written just before).  It is launched as a programmatic dependent of the GEMM
// and waits (griddepcontrol.wait) for that grid to complete before it reads a plane.
#include <cuda_fp16.h>

#include "qgemm_common.cuh"
#include "qgemm_internal.h"
#include "qgemm_ptx.cuh"

namespace {

using namespace qg;

constexpr int THREADS = 256;

__global__ void __launch_bounds__(THREADS)
splitk_reduce_kernel(const float *__restrict__ P, int splits, int64_t plane, int64_t ldp, int M,
                     int N, __half *__restrict__ C, int64_t ldc, int c_vec, int epi) {
    griddep_wait();
    const int groups = (N + 3) / 4;                 // 4-column groups per row
    const int64_t total = static_cast<int64_t>(M) * groups;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * THREADS + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * THREADS) {
        const int m = static_cast<int>(i / groups);
        const int n0 = 4 * static_cast<int>(i - static_cast<int64_t>(m) * groups);
        const float *p = P + static_cast<int64_t>(m) * ldp + n0;
        float4 acc = __ldcg(reinterpret_cast<const float4 *>(p));
        // eight planes' loads in flight at a time, then their sums in split order
        for (int s0 = 1; s0 < splits; s0 += 8) {
            float4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (s0 + j < splits) v[j] = __ldcg(reinterpret_cast<const float4 *>(p + (s0 + j) * plane));
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (s0 + j < splits) {
                    acc.x += v[j].x;
                    acc.y += v[j].y;
                    acc.z += v[j].z;
                    acc.w += v[j].w;
                }
            }
        }
        float x[4] = {acc.x, acc.y, acc.z, acc.w};
        __half *crow = C + static_cast<int64_t>(m) * ldc + n0;
        const int nv = min(4, N - n0);                 // columns of this group inside C
        const bool v4 = c_vec != 0 && nv == 4;
        if (epi & EPI_ACC_BIT) {
            if (v4) {
                const uint2 w = *reinterpret_cast<const uint2 *>(crow);
                const __half2 lo = *reinterpret_cast<const __half2 *>(&w.x);
                const __half2 hi = *reinterpret_cast<const __half2 *>(&w.y);
                x[0] += __low2float(lo);
                x[1] += __high2float(lo);
                x[2] += __low2float(hi);
                x[3] += __high2float(hi);
            } else {
                for (int j = 0; j < nv; ++j) x[j] += __half2float(crow[j]);
            }
        }
        if (epi & EPI_RELU_BIT) {
#pragma unroll
            for (int j = 0; j < 4; ++j) x[j] = fmaxf(x[j], 0.0f);
        }
        if (v4) {
            *reinterpret_cast<uint2 *>(crow) = make_uint2(pack_f16x2(x[0], x[1]), pack_f16x2(x[2], x[3]));
        } else {
            for (int j = 0; j < nv; ++j) crow[j] = __float2half_rn(x[j]);
        }
    }
}

}  // namespace

namespace qgi {

cudaError_t launch_splitk_reduce(const float *P, int splits, int64_t ldp, int M, int N, __half *C,
                                 int64_t ldc, const LaunchCtx &ctx) {
    const int64_t total = static_cast<int64_t>(M) * ((N + 3) / 4);
    if (total == 0) return cudaSuccess;
    int64_t blocks = (total + THREADS - 1) / THREADS;
    const int64_t cap = static_cast<int64_t>(ctx.num_sms) * 8;
    if (blocks > cap) blocks = cap;
    const int c_vec = (reinterpret_cast<uintptr_t>(C) % 8 == 0 && ldc % 4 == 0) ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel, P, splits,
                              static_cast<int64_t>(M) * ldp, ldp, M, N, C, ldc, c_vec, ctx.epi);
}

}  // namespace qgi
