// qgemm_internal.h -- host-side internals shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "qgemm.h"

// The view behind the opaque handle: borrowed device pointers plus shape.
struct qgemm_tensor {
    int32_t dtype;
    int64_t rows;
    int64_t k;
    const uint8_t *data;
    int64_t ld;          // bytes between rows of the data plane
    const uint8_t *scales;
    int64_t lds;         // bytes between rows of the scale plane
};

namespace qgi {

// Epilogue flags (LaunchCtx::epi): C = relu?( acc [+ C_old] ), one fp16 rounding at the end.
constexpr int EPI_ACCUMULATE = 1;   // add the existing C (fp16) to the fp32 accumulator
constexpr int EPI_RELU = 2;         // max(x, +0) before rounding

struct LaunchCtx {
    cudaStream_t stream;
    unsigned *err;        // device error word
    uint64_t timeout_ns;  // bound on every device-side wait
    int num_sms;
    int device;
    int epi = 0;          // EPI_* flags of the output epilogue
};

// Records a formatted message for qgemm_last_error_message() and returns `s`.
qgemm_status fail(qgemm_status s, const char *fmt, ...);

// Encode a 2-D tiled TMA descriptor (inner dimension first).  Returns false on failure.
bool encode_tma_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t inner,
                   uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                   uint32_t box_outer, CUtensorMapSwizzle swizzle);

// Encode a 3-D tiled TMA descriptor (dimension 0 innermost; strides of dimensions 1 and 2).
bool encode_tma_3d(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t d0,
                   uint64_t d1, uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes,
                   uint32_t box0, uint32_t box1, uint32_t box2, CUtensorMapSwizzle swizzle);

// Kernel launchers (one per translation unit).  Arguments are already validated.
// allow_split = false keeps the one-CTA route to one pass (no K split, hence no scratch).
cudaError_t launch_mxfp8(const qgemm_tensor *A, const qgemm_tensor *B, __half *C, int64_t ldc,
                         const LaunchCtx &ctx, bool *encode_ok, bool allow_split = true);
// Device scratch a launch_mxfp8 call (allow_split = true) takes from the pool, in bytes.
size_t mxfp8_scratch_bytes(const qgemm_tensor *A, const qgemm_tensor *B, int num_sms);
// Split-K reduction: C[m, n] = fp16_rn( relu?( sum_{s = 0 .. splits-1, in order} P[s][m][n]
// [+ C_old[m, n]] ) ) under ctx.epi, P holding `splits` planes of M rows x ldp floats (ldp a
// multiple of 4, P 16-byte aligned).  Launched as a programmatic dependent of the GEMM that
// writes P.
cudaError_t launch_splitk_reduce(const float *P, int splits, int64_t ldp, int M, int N, __half *C,
                                 int64_t ldc, const LaunchCtx &ctx);
// CTA-pair MXFP8 path: scales are repacked into `scratch` (mxfp8_pair_scratch_bytes bytes,
// 256-byte aligned device memory that stays untouched by anything else until the GEMM is done).
bool mxfp8_pair_eligible(const qgemm_tensor *A, const qgemm_tensor *B);
size_t mxfp8_pair_scratch_bytes(const qgemm_tensor *A, const qgemm_tensor *B);
cudaError_t launch_mxfp8_pair(const qgemm_tensor *A, const qgemm_tensor *B, __half *C,
                              int64_t ldc, void *scratch, const LaunchCtx &ctx, bool *encode_ok);

// The two halves of launch_mxfp8_pair, for callers that repack an operand once and reuse it:
// the repack of one view's scale plane into `out` (mxfp8_pack_bytes(T) bytes, 256-byte aligned),
// and the CTA-pair GEMM on planes repacked that way.
size_t mxfp8_pack_bytes(const qgemm_tensor *T);
cudaError_t launch_mxfp8_sf_pack(const qgemm_tensor *T, void *out, const LaunchCtx &ctx);
cudaError_t launch_mxfp8_pair_packed(const qgemm_tensor *A, const qgemm_tensor *B, __half *C,
                                     int64_t ldc, const void *packA, const void *packB,
                                     const LaunchCtx &ctx, bool *encode_ok);

// MXFP4 (E2M1) GEMM on CTA pairs, same pipeline and scratch contract as launch_mxfp8_pair.
size_t mxfp4_scratch_bytes(const qgemm_tensor *A, const qgemm_tensor *B);
cudaError_t launch_mxfp4_pair(const qgemm_tensor *A, const qgemm_tensor *B, __half *C,
                              int64_t ldc, void *scratch, const LaunchCtx &ctx, bool *encode_ok);

// Stream-ordered scratch from the library's per-device memory pool (memory is kept in the pool
// between calls, so steady-state calls do not reach the driver's allocator).
cudaError_t scratch_alloc(size_t bytes, const LaunchCtx &ctx, void **p);
cudaError_t scratch_free(void *p, const LaunchCtx &ctx);

// Launch context on the current device (SM count, error word, wait bound), for entry points
// defined outside qgemm_api.cu.
qgemm_status launch_ctx(void *stream, LaunchCtx *ctx);
cudaError_t launch_gemm_f16(const __half *A, int64_t lda, const __half *B, int64_t ldb,
                            __half *C, int64_t ldc, int M, int N, int K, const LaunchCtx &ctx,
                            bool *encode_ok);
cudaError_t launch_w4a16(const __half *A, int64_t lda, int M, const qgemm_tensor *W, __half *C,
                         int64_t ldc, const LaunchCtx &ctx, bool *encode_ok);
// Exact recomputation of the outlier rows of an int4 view (a nonzero weight in a block whose
// UE8M0 byte is outside 103..139 and not 255) after launch_w4a16 on the same stream, under the
// same ctx.epi (w4a16_outlier.cu).
cudaError_t launch_w4a16_outliers(const __half *A, int64_t lda, int M, const qgemm_tensor *W,
                                  __half *C, int64_t ldc, const LaunchCtx &ctx);
// CTA-pair W4A16 with the dequantised weights in TMEM (w4a16_pair.cu).
bool w4a16_pair_eligible(int M, const qgemm_tensor *W);
cudaError_t launch_w4a16_pair(const __half *A, int64_t lda, int M, const qgemm_tensor *W,
                              __half *C, int64_t ldc, const LaunchCtx &ctx, bool *encode_ok);
// int4 weights [N, K] (packed, row stride ldw bytes) with fp16 block-32 scales [N, K/32] (row
// stride lds_elems), on the CTA-pair kernel: K % 256 == 0, W and scales 16-byte aligned rows.
cudaError_t launch_w4a16_f16s(const __half *A, int64_t lda, int M, const uint8_t *W_int4,
                              int64_t ldw, const __half *scales, int64_t lds_elems, int N, int K,
                              __half *C, int64_t ldc, const LaunchCtx &ctx, bool *encode_ok);
cudaError_t launch_w8_gemv(const __half *X, int64_t ldx, int M, const qgemm_tensor *W,
                           __half *Y, int64_t ldy, const LaunchCtx &ctx, bool *encode_ok);
// Fused attention, head dimension 128: O = softmax(scale Q K^T) V per head (attention.cu).
struct AttnArgs {
    const __half *Q, *K, *V;
    __half *O;
    int64_t q_hs, q_rs, k_hs, k_rs, v_hs, v_rs, o_hs, o_rs;   // strides in elements
    int BH, Lq, Lk;
    float scale;
};
cudaError_t launch_attention(const AttnArgs &a, const LaunchCtx &ctx, bool *encode_ok);
cudaError_t launch_dequant(const qgemm_tensor *t, float *out, const LaunchCtx &ctx);
cudaError_t launch_fill_zero_f16(__half *C, int64_t ldc, int64_t M, int64_t N,
                                 const LaunchCtx &ctx);
// K = 0: C = relu?(0 [+ C_old]) under ctx.epi.
cudaError_t launch_empty_sum_epilogue(__half *C, int64_t ldc, int64_t M, int64_t N,
                                      const LaunchCtx &ctx);
cudaError_t launch_selftest_wait(uint64_t timeout_ns, const LaunchCtx &ctx);
cudaError_t launch_clock_probe(uint64_t window_ns, uint64_t *out, const LaunchCtx &ctx);

}  // namespace qgi
