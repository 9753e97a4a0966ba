/*
 * qgemm.h -- C ABI of the block-scaled quantized GEMM library for GB300 (sm_103a).
 *
 * The operation is the quantized matmul2d of "TensorOps: quantized matmul, cooperative tensors,
 * and the neural accelerator" (section "Quantized matmul2d -- and the custom-format escape
 * hatch"): the quantized product uses the same call shape as the fp16 one, the operands carry a
 * data plane plus a scale plane, and the library dequantises on the fly.  Every product below is
 *
 *     C[m, n] = fp16_rn( sum_k deq(A)[m, k] * deq(B)[n, k] )       (fp32 accumulation)
 *
 * with deq(X)[r, k] = decode(X.data[r, k]) * 2^(X.scales[r, k / 32] - 127).  The output is always
 * overwritten ("mode multiply", same page, section "The real matmul2d API").
 *
 * Conventions that hold for every call:
 *   - All data, scale and output pointers are DEVICE pointers owned by the caller (host pointers
 *     for qgemm_mxfp8_host).  The library never frees or retains them; a qgemm_tensor only
 *     borrows pointers.  The device memory the library takes for itself is stated at each call
 *     that uses it: the scale scratch of the CTA-pair block-scaled GEMMs and the fp32 partial
 *     planes of a split K (both from a per-device pool), the attention workspace, the staging
 *     buffers of qgemm_mxfp8_host, the fixed array of qgemm_mxfp8_noalloc.
 *   - Results are repeatable: the same inputs on the same GPU give the same output bits (every
 *     sum is taken in a fixed order, independent of timing).
 *   - Matrices are row-major with the reduction dimension K contiguous ("K-major"), except the
 *     right operand of gemm_f16, which is B[K, N] row-major (N contiguous).
 *   - Row strides are given in BYTES for qgemm_tensor planes and in ELEMENTS for plain fp16
 *     matrices (lda, ldb, ldc, ldx, ldy).
 *   - A stream argument is a cudaStream_t passed as void* (NULL = legacy default stream).  Compute
 *     calls only validate and enqueue; they return before the GPU finishes.  Errors found on the
 *     host are returned before anything is enqueued (nothing is written).  A failed launch
 *     returns QGEMM_ERR_CUDA.
 *   - Every device-side wait is bounded.  A kernel that gives up records a code in a device
 *     error word that qgemm_poll_device_error() reads; its outputs are then unspecified.
 *   - The library caches per-device addresses (the error word, the fixed array of
 *     qgemm_mxfp8_noalloc) in the device's primary context: after cudaDeviceReset, or any other
 *     teardown of that context, the library must not be called again in the same process.
 */
#ifndef QGEMM_H
#define QGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QGEMM_OK = 0,
    QGEMM_ERR_INVALID_ARG = 1,       /* null pointer, negative size, inconsistent shapes       */
    QGEMM_ERR_UNSUPPORTED_SHAPE = 2, /* a size the kernels do not take (e.g. K % 32 != 0)      */
    QGEMM_ERR_MISALIGNED = 3,        /* pointer or stride alignment below what the kernel needs */
    QGEMM_ERR_UNSUPPORTED_DTYPE = 4, /* wrong data type for the call, or block size != 32     */
    QGEMM_ERR_CUDA = 5,              /* a CUDA runtime/driver call failed (see last message)   */
    QGEMM_ERR_TIMEOUT = 6            /* a kernel's bounded wait ran out (device error word)    */
} qgemm_status;

typedef enum {
    QGEMM_F16 = 0,   /* IEEE binary16, no scale plane                                        */
    QGEMM_E4M3 = 1,  /* FP8 E4M3 (OCP, no infinity), one byte per element                    */
    QGEMM_INT8 = 2,  /* two's complement int8, one byte per element                          */
    QGEMM_INT4 = 3,  /* two's complement int4, two per byte, even k in the low nibble        */
    QGEMM_E2M1 = 4   /* FP4 E2M1 (sign, 2 exponent bits with bias 1, 1 mantissa bit; values
                        0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives), two per byte, even k in
                        the low nibble                                                        */
} qgemm_dtype;

/* Opaque, host-side, NON-owning view of one quantized matrix [rows, k]. */
typedef struct qgemm_tensor qgemm_tensor;

/* Library version, (major << 16) | minor. */
int32_t qgemm_version(void);

/* 1 in the debug build (libqgemm_debug.so, compiled with QGEMM_DEBUG: every kernel checks its own
 * index arithmetic and reports a failed check as bit 32 of the device error word, see
 * qgemm_poll_device_error), 0 in the release build.  The pages have no counterpart: it lets a
 * test confirm which build it runs. */
int32_t qgemm_debug_build(void);

/* Create a view of a quantized matrix: data plane plus UE8M0 scale plane.
 * Passage: "TensorOps: quantized matmul ...", section "Scale planes: one MTLTensor = data +
 * scales" (one object carries the data plane and an auxiliary plane of block scales; the block
 * factors give how many data elements share one scale) and "Optimize custom machine learning
 * operations with Metal tensors", section "Creating quantized tensors with scale factors" (a
 * failed creation reports an error and yields no tensor).  The scale type must be UE8M0 and the
 * block 32 along K by 1 along rows (same first page, "Kernel-phase findings", fact 2).
 *   out            receives the new view; set to NULL on any error.
 *   dt             element type of the data plane.
 *   rows, k        logical shape [rows, k]; k is the contiguous (reduction) dimension.
 *   data           device pointer to element (0, 0); row r starts at data + r * data_row_stride_bytes.
 *                  int4, E2M1: element (r, k) is nibble (k & 1) of byte k / 2 of row r.
 *   scales_ue8m0   device pointer to the [rows, ceil(k / 32)] UE8M0 scale plane; scale (r, b) at
 *                  scales_ue8m0 + r * scale_row_stride_bytes + b.  Must be NULL for QGEMM_F16 and
 *                  non-NULL for the other types.
 *   block_k        must be 32 (QGEMM_ERR_UNSUPPORTED_DTYPE otherwise; ignored for QGEMM_F16).
 * Errors: QGEMM_ERR_INVALID_ARG (null out/data, negative sizes, strides shorter than a row),
 *         QGEMM_ERR_UNSUPPORTED_SHAPE (k % 32 != 0 for a scaled type),
 *         QGEMM_ERR_UNSUPPORTED_DTYPE (unknown dtype, block_k != 32, scales present for F16). */
qgemm_status qgemm_create_tensor(qgemm_tensor **out, qgemm_dtype dt, int64_t rows, int64_t k,
                                 const void *data, int64_t data_row_stride_bytes,
                                 const uint8_t *scales_ue8m0, int64_t scale_row_stride_bytes,
                                 int32_t block_k);

/* View of rows [row0, row0 + nrows) and columns [k0, k0 + nk) of t; data and scale planes are
 * sliced together so the sub-view's block grid stays aligned ("TensorOps: quantized matmul ...",
 * section "Scale planes ...": slicing a quantized tensor slices both planes, respecting the block
 * size).  k0 must be a multiple of 32 for scaled types (and even for int4); the slice must lie
 * inside t.  The new view borrows the same memory and is independent of t's lifetime.
 * Errors: QGEMM_ERR_INVALID_ARG (null, out of range), QGEMM_ERR_UNSUPPORTED_SHAPE (k0 or nk not
 * block-aligned). */
qgemm_status qgemm_tensor_slice(const qgemm_tensor *t, int64_t row0, int64_t nrows, int64_t k0,
                                int64_t nk, qgemm_tensor **out);

/* Free the view (host memory only; never touches device memory).  NULL is a no-op.
 * Passage: the pages have no counterpart (a Metal tensor is reference-counted); a view here is a
 * plain host object, so its owner frees it. */
void qgemm_destroy_tensor(qgemm_tensor *t);

/* Read back a view's fields (any out-pointer may be NULL). */
qgemm_status qgemm_tensor_info(const qgemm_tensor *t, int32_t *dtype, int64_t *rows, int64_t *k,
                               const void **data, int64_t *data_row_stride_bytes,
                               const uint8_t **scales, int64_t *scale_row_stride_bytes);

/* MXFP8 GEMM: C[M, N] = fp16_rn(sum_k deq(A)[m, k] * deq(B)[n, k]), fp32 accumulation.
 * Passage: "Optimize custom machine learning operations with Metal tensors", sections "Shader
 * MXFP8 tensor types" and "Slicing and quantized matmul" (E4M3 data with a UE8M0 block-32 scale
 * plane fed straight into matmul2d), with the right operand stored transposed, i.e. [N, K]
 * ("TensorOps: quantized matmul ...", "Kernel-phase findings", fact 2).
 *   A   QGEMM_E4M3 view [M, K];  B   QGEMM_E4M3 view [N, K] (same K).
 *   C   device fp16 [M, N] with row stride ldc elements (ldc >= N).
 * Requirements: K % 32 == 0; data pointers and byte strides 16-byte aligned; scale planes any
 * alignment; C 2-byte aligned (16-byte aligned C and ldc % 8 == 0 take the vector stores).  Any
 * M, N >= 0 (ragged tiles are masked); M or N == 0 writes nothing; K == 0 writes zeros.
 * Scratch: when M > 128 and N > 128 the call runs on CTA pairs and first rewrites both scale
 * planes into the order the tensor cores read them, in (2 ceil(M/256) + 2 ceil(N/256)) *
 * ceil(K/128) * 512 bytes of device scratch taken from a library-owned per-device memory pool
 * with cudaMallocFromPoolAsync on `stream` and handed back with cudaFreeAsync on the same stream
 * after the GEMM (two kernel launches).  The pool keeps its memory between calls, so steady-state
 * calls do not reach the driver's allocator; it is released at process exit.  Otherwise (M or
 * N <= 128) one CTA computes each 128 x 256 (128 x 128 for N <= 128) output tile; when there are
 * at most half as many tiles as SMs, K is split: S = min(SMs / tiles, ceil(K / 512)) CTAs per
 * tile each sum a range of whole 512-wide slices of K into an fp32 partial plane of pooled
 * scratch (S * M * ceil(N / BN) * BN * 4 bytes, BN the tile width), and a second kernel adds the
 * S planes in a fixed order and writes C (so the bits depend on S, which depends on the GPU's SM
 * count, and remain repeatable).  qgemm_mxfp8_scratch_bytes tells how much a call takes.
 * Errors: INVALID_ARG, UNSUPPORTED_DTYPE, UNSUPPORTED_SHAPE, MISALIGNED (nothing enqueued); CUDA
 * (including a failed scratch allocation). */
qgemm_status qgemm_mxfp8(const qgemm_tensor *A, const qgemm_tensor *B, void *C, int64_t ldc,
                         void *stream);

/* The device scratch one qgemm_mxfp8 call with these views takes from the library's pool on the
 * current device, in bytes (0: none): the repacked scale planes on the CTA-pair route, or the
 * fp32 partial planes of a K split on the one-CTA route (both described at qgemm_mxfp8).  No
 * counterpart on the pages: it lets a caller that manages device memory itself leave room for the
 * call (or take qgemm_mxfp8_noalloc).  Nothing is launched.
 *   bytes  host pointer receiving the size.
 * Errors: INVALID_ARG (NULL view or bytes, K mismatch), UNSUPPORTED_DTYPE (not E4M3 views), CUDA
 * (the device cannot be queried). */
qgemm_status qgemm_mxfp8_scratch_bytes(const qgemm_tensor *A, const qgemm_tensor *B,
                                       int64_t *bytes);

/* qgemm_mxfp8 without any device allocation.  The paper has no counterpart: this entry point
 * exists for callers that cannot let a library allocate device memory while they run -- a serving
 * process that reserves all device memory up front for its own allocator, or a latency-critical
 * path that cannot risk an allocation that blocks or fails in the middle of a request.
 * Same arguments, layouts, results and errors as qgemm_mxfp8.  Where qgemm_mxfp8 takes pooled
 * scratch for the repacked scale planes (M > 128 and N > 128), this call uses a fixed 8 MiB
 * device array compiled into the library instead (held, once placed, on each device until exit)
 * and makes no cudaMalloc, pool allocation or other allocating call.  M or N <= 128 runs the
 * one-CTA kernel of qgemm_mxfp8 in one pass over K, which needs no scratch; where qgemm_mxfp8
 * splits K for such a shape the two calls sum in different orders, and their outputs can differ
 * in the last bit (both within the same bound of the exact product).
 * Limits and rules:
 *   - a shape whose repacked scales need more than 8 MiB ((2 ceil(M/256) + 2 ceil(N/256)) *
 *     ceil(K/128) * 512 bytes, e.g. more than M = N = 16384 at K = 8192) is rejected with
 *     QGEMM_ERR_UNSUPPORTED_SHAPE and nothing is launched;
 *   - all calls on one device share the array: calls that overlap on the GPU race on it and give
 *     wrong results -- issue them on one stream or synchronise between them;
 *   - the array keeps the last call's contents; every byte a call reads is first rewritten by it;
 *   - the first call on each device looks up the array's device address (cudaGetSymbolAddress,
 *     with that device current) and caches it; make that first call before any stream capture;
 *   - under CUDA's lazy module loading (the default) that first lookup is also when the driver
 *     places the 8 MiB in the device's memory: a caller that reserves all remaining device memory
 *     for itself makes one call on each device before it does so. */
qgemm_status qgemm_mxfp8_noalloc(const qgemm_tensor *A, const qgemm_tensor *B, void *C,
                                 int64_t ldc, void *stream);

/* MXFP4 GEMM: C[M, N] = fp16_rn(sum_k deq(A)[m, k] * deq(B)[n, k]), fp32 accumulation, with
 * deq(x)[r, k] = e2m1(x[r, k]) * 2^(scale[r, k / 32] - 127).
 * Passage: "TensorOps: quantized matmul ...", section "Quantized dtype support matrix" (fp4 data
 * fed natively to matmul2d, with the MX block scale factors in FP8 E8M0 as the scale plane) and
 * "Optimize custom machine learning operations with Metal tensors", sections on native quantized
 * types (4-bit floating point added beside FP8) and on multi-plane tensors (one E8M0 scale per
 * block of the data plane); the right operand stored transposed, [N, K], as for qgemm_mxfp8.
 *   A   QGEMM_E2M1 view [M, K];  B   QGEMM_E2M1 view [N, K] (same K), scales UE8M0 per 32.
 *   C   device fp16 [M, N] with row stride ldc elements (ldc >= N).
 * Requirements: K % 32 == 0; data pointers and byte strides 16-byte aligned; scale planes any
 * alignment; C 2-byte aligned.  Any M, N >= 0 (every shape runs on CTA pairs, ragged tiles
 * masked); M or N == 0 writes nothing; K == 0 writes zeros.
 * Scratch: both scale planes are first rewritten into the order the tensor cores read them, in
 * (2 ceil(M/256) + 2 ceil(N/256)) * ceil(K/256) * 1024 bytes of device scratch taken from the
 * library's per-device pool on `stream` (as qgemm_mxfp8; two kernel launches).
 * Errors: INVALID_ARG, UNSUPPORTED_DTYPE, UNSUPPORTED_SHAPE, MISALIGNED (nothing enqueued); CUDA
 * (including a failed scratch allocation). */
qgemm_status qgemm_mxfp4(const qgemm_tensor *A, const qgemm_tensor *B, void *C, int64_t ldc,
                         void *stream);

/* qgemm_mxfp8 on host memory: A and B are views whose data and scale planes are in host memory
 * (page-locked memory lets the copies run asynchronously; pageable memory works but the copies
 * then stage through the driver), C is host fp16 [M, N] with row stride ldc elements.  The pages
 * have no counterpart: this is the end-to-end form of the product for a caller whose operands
 * live on the host.  One call uploads both operands, runs the GEMM of qgemm_mxfp8 and downloads
 * C, overlapping the three: B first, then A in row chunks; each chunk's product starts when that
 * chunk has landed and each finished chunk of C is downloaded while the next one computes.
 * Ordering: everything is ordered after the work already on `stream`, and `stream` completes
 * only after C is on the host; calls on one stream therefore run one after another, while calls
 * on different streams overlap (the uploads of one with the downloads of another).  The host
 * planes must not be modified, nor C read, before `stream` has completed the call.
 * Device memory: two buffer sets per device, grown to the largest shape seen, held until exit
 * (A + B + scales + C: 272 MB each at M = N = K = 8192), plus the scratch of qgemm_mxfp8.
 * Requirements and errors: as qgemm_mxfp8 (no alignment rule for the host planes); CUDA also for
 * a failed copy or allocation. */
qgemm_status qgemm_mxfp8_host(const qgemm_tensor *A, const qgemm_tensor *B, void *C, int64_t ldc,
                              void *stream);

/* fp16 GEMM: C[M, N] = fp16_rn(A[M, K] @ B[K, N]), fp32 accumulation, all row-major fp16.
 * Passage: "TensorOps: quantized matmul ...", "VALIDATED ON M4 MAX" (kernel M0, half x half ->
 * half) and "TileLang Metal Backend Internals", section 1 (fp16 input, fp32 accumulation, fp16
 * output cast on store).
 * Requirements: A, B, C 16-byte aligned; lda, ldb, ldc multiples of 8 elements; lda >= K,
 * ldb >= N, ldc >= N.  Any M, N, K >= 0 (ragged tiles masked; K == 0 writes zeros).
 * Scratch: M > 128 and N > 128 run on CTA pairs and take none.  Otherwise one CTA computes each
 * 128 x 256 (128 x 128 for N <= 128) tile, and when there are at most half as many tiles as SMs
 * K is split as for qgemm_mxfp8: S = min(SMs / tiles, ceil(K / 512)) CTAs per tile write fp32
 * partial planes into S * M * ceil(N / BN) * BN * 4 bytes taken from the library's pool on
 * `stream` (and handed back after the reduction kernel that adds them in a fixed order).
 * Errors: INVALID_ARG, MISALIGNED (nothing enqueued); CUDA (including a failed scratch
 * allocation). */
qgemm_status gemm_f16(const void *A, int64_t lda, const void *B, int64_t ldb, void *C,
                      int64_t ldc, int64_t M, int64_t N, int64_t K, void *stream);

/* Weight-only int4 GEMM (prefill): C[M, N] = fp16_rn(sum_k A[m, k] * deq(W)[n, k]).
 * Passage: "TensorOps: quantized matmul ...", "Revised kernel strategy" and "M2 = block-32 fp16
 * scaling" (dequantise each 32-block of the int4 weight with its scale, then feed the half x half
 * matmul, accumulating across blocks), with the int4 packing of "VALIDATED ON M4 MAX", fact 5.
 *   A   device fp16 [M, K], row stride lda elements.
 *   W   QGEMM_INT4 view [N, K] with UE8M0 scales [N, K / 32].
 *   C   device fp16 [M, N], row stride ldc.
 * Numerics: the defined product for every scale byte.  Inside the fold window 103 <= e <= 139
 * each weight becomes the fp16 value q * 2^(e - 127) (exact: |w| lies in [2^-24, 2^15]) and the
 * tensor cores form the fp32 sum.  Byte 255 is NaN and makes the row's outputs NaN (q * NaN is
 * NaN for every q, zero included).  A block with any other byte contributes exactly zero when
 * its weights are all zero; a weight row with a nonzero weight in such a block (an outlier row)
 * is computed again by a second kernel on the same stream: fp32 partial sums per 32-block, each
 * times its 2^(e - 127) and summed in fp64, one fp16 rounding (with the epilogue of the _ex call
 * applied to that sum).  Outlier rows cost M * K fused multiply-adds each on the CUDA cores; the
 * second kernel is launched by every call and, with no outlier row, only reads the scale plane.
 * Scratch: with N > 128, K % 512 == 0 and 16-byte aligned scale rows the product runs on CTA
 * pairs (256 weight rows x 256 tokens per pair tile); when the tiles fill at most half of the
 * pairs (a few tokens against many weight rows) and C is not accumulated (qgemm_w4a16_ex), each
 * tile's K is split in whole 512-wide slices over S = min(pairs / tiles, K / 512) pairs, whose
 * fp32 partial planes (S * M * ceil(N / 256) * 256 * 4 bytes, from the library's pool on
 * `stream`) a reduction kernel adds in a fixed order before the outlier-row kernel runs.
 * Requirements: K % 64 == 0; A, C 16-byte aligned; lda, ldc multiples of 8; W data 16-byte
 * aligned with a 16-byte multiple row stride; any M, N.
 * Errors: INVALID_ARG, UNSUPPORTED_DTYPE, UNSUPPORTED_SHAPE, MISALIGNED; CUDA (including a
 * failed scratch allocation). */
qgemm_status qgemm_w4a16(const void *A_f16, int64_t lda, int64_t M, const qgemm_tensor *W,
                         void *C_f16, int64_t ldc, void *stream);

/* Custom-format escape hatch: int4 weights with arbitrary fp16 scales per block of 32 along K.
 * C[M, N] = fp16_rn(sum_k A[m, k] * w[n, k]),  w[n, k] = fp16_rn(q[n, k] * S[n, k / 32]),
 * fp32 accumulation.
 * Passage: "TensorOps: quantized matmul ...", sections "Two facts ..." (fact 2: the native scale
 * plane takes only E8M0, so arbitrary fp16 block scales cannot ride on a tensor view), "Revised
 * kernel strategy" and "M2 = block-32 fp16 scaling" (each weight of a 32-block dequantised into
 * half as its int4 value times the block's fp16 scale, then the half x half matmul with fp32
 * accumulation).  The dequantised weight is the half nearest to q * s (ties to even): exactly
 * one rounding, as the recipe's half multiply gives.  Raw pointers, no view: the format is
 * outside the native tensor type.
 *   A        device fp16 [M, K], row stride lda elements.
 *   W_int4   device int4 [N, K], two per byte (even k in the low nibble), row stride ldw_bytes.
 *   scales   device fp16 [N, K / 32], row stride lds elements; any fp16 values (inf and NaN
 *            propagate as the half multiply gives).
 *   C        device fp16 [M, N], row stride ldc elements.
 * Requirements: K % 256 == 0; A 16-byte aligned with lda % 8 == 0; W 16-byte aligned with
 * ldw_bytes % 16 == 0; scales 16-byte aligned with lds % 8 == 0; C 2-byte aligned (16-byte
 * aligned C with ldc % 8 == 0 takes TMA stores); any M, N >= 0 (ragged tiles masked; K == 0
 * writes zeros).  Runs on CTA pairs for every shape, with K split over several pairs as for
 * qgemm_w4a16 when the tiles fill at most half of them and C is not accumulated (pooled fp32
 * partial planes, reduced in a fixed order).
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED (nothing enqueued); CUDA (including a
 * failed scratch allocation). */
qgemm_status qgemm_w4a16_f16s(const void *A_f16, int64_t lda, int64_t M, const void *W_int4,
                              int64_t ldw_bytes, const void *scales_f16, int64_t lds, int64_t N,
                              int64_t K, void *C_f16, int64_t ldc, void *stream);

/* Decode GEMV with int8 weights: Y[m, n] = fp16_rn(sum_k X[m, k] * deq(W)[n, k]), 1 <= M <= 16.
 * Passage: "TensorOps: quantized matmul ...", section "Why this matters here" (decode is bound
 * by memory bandwidth; int8 weights are read at int8 cost) and "VALIDATED ON M4 MAX" (kernel
 * M1a, half x int8 -> half).  Each 32-block partial sum is scaled by its power of two in fp32,
 * so every scale byte 0..254 is handled exactly.
 *   X   device fp16 [M, K], row stride ldx elements.
 *   W   QGEMM_INT8 view [N, K] with UE8M0 scales [N, K / 32].
 *   Y   device fp16 [M, N], row stride ldy elements.
 * Requirements: 1 <= M <= 16; K % 32 == 0; X 16-byte aligned, ldx multiple of 8; W data and row
 * stride 16-byte aligned; scale plane any alignment; Y 2-byte aligned.
 * Errors: INVALID_ARG, UNSUPPORTED_DTYPE, UNSUPPORTED_SHAPE, MISALIGNED; CUDA. */
qgemm_status qgemm_w8_gemv(const void *X_f16, int64_t ldx, int64_t M, const qgemm_tensor *W,
                           void *Y_f16, int64_t ldy, void *stream);

/* Fused attention forward: for every head h and query row i,
 *   O[h, i, :] = sum_j softmax_j(scale * <Q[h, i, :], K[h, j, :]>) V[h, j, :],
 * fp16 Q, K, V and O, scores and the softmax in fp32, P = exp(s - max) rounded to fp16 for the
 * second product, fp32 accumulation, one fp16 rounding of O.  No mask.
 * Passage: "TensorOps: quantized matmul ...", section "FlashAttention on TensorOps (the recipe)"
 * and "Optimize custom machine learning operations with Metal tensors", section on FlashAttention
 * with cooperative tensors (Q K^T, the row maximum with initial value -infinity, exp of each
 * score minus it, times V, in one kernel with the intermediate never written to memory; the
 * softmax is normalised by its row sum, the scale is the caller's, e.g. 1/sqrt(d)).
 *   Q, O     device fp16 [BH, Lq, d];  K, V  device fp16 [BH, Lk, d]; element (h, i, c) of X at
 *            X + h * x_head_stride + i * x_row_stride + c (strides in elements).
 * Requirements: d == 128; Lk >= 1; BH <= 65535; scale finite and > 0; every base 16-byte aligned
 * and every stride a multiple of 8 (and non-negative); O's rows must not overlap: heads outside
 * rows (row stride >= d, head stride >= Lq * row stride) or rows outside heads (head stride >= d,
 * row stride >= BH * head stride, as in a [batch, L, heads, d] buffer).  BH == 0 or Lq == 0 does
 * nothing.
 * Launch: one cooperative kernel of up to one CTA per SM (every CTA resident at once: CTAs merge
 * the rows of units they share), preceded, when work ranges cut units, by a memset of the flags
 * in a stream-ordered workspace of about 133 KB per CTA taken from the library's pool and freed
 * after the launch.  The result does not depend on the stream's other work and repeats bit for
 * bit for the same inputs and SM count.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED (nothing enqueued); CUDA (including a
 * cooperative launch the device cannot make resident). */
qgemm_status qgemm_attention_f16(const void *Q, const void *K, const void *V, void *O, int64_t BH,
                                 int64_t Lq, int64_t Lk, int64_t d, int64_t q_head_stride,
                                 int64_t q_row_stride, int64_t k_head_stride, int64_t k_row_stride,
                                 int64_t v_head_stride, int64_t v_row_stride,
                                 int64_t o_head_stride, int64_t o_row_stride, float scale,
                                 void *stream);

/* ---------------------------------------------------------------- fused output epilogue
 * C = relu?( A*B [+ C_old] ): the product's fp32 accumulator plus, when `accumulate` is set,
 * the existing fp16 output (read before it is overwritten), then, when `relu` is set,
 * max(x, +0); one fp16 round-to-nearest-even at the end.
 * Passages: "TensorOps: quantized matmul ...", section "The real matmul2d API" (the op's mode is
 * multiply or multiply_accumulate, the latter computing C = A*B + C); "Running inline ML
 * operations in a shader with Metal 4", section "Combine an element-wise function" (a ReLU
 * postfix applied to the product's elements before they are stored, in the same dispatch).
 * Each _ex call takes the arguments of the call it extends plus `epilogue` (NULL = plain store);
 * its fields must be 0 or 1 (QGEMM_ERR_INVALID_ARG otherwise).  With accumulate set the output
 * must hold valid fp16 data; K == 0 then leaves relu?(C_old).  Errors as the plain calls. */
typedef struct qgemm_epilogue {
    int32_t accumulate;   /* 1: add the existing output (matmul2d multiply_accumulate) */
    int32_t relu;         /* 1: max(x, +0) before the rounding */
} qgemm_epilogue;

qgemm_status qgemm_mxfp8_ex(const qgemm_tensor *A, const qgemm_tensor *B, void *C, int64_t ldc,
                            const qgemm_epilogue *epilogue, void *stream);
qgemm_status qgemm_mxfp4_ex(const qgemm_tensor *A, const qgemm_tensor *B, void *C, int64_t ldc,
                            const qgemm_epilogue *epilogue, void *stream);
qgemm_status gemm_f16_ex(const void *A, int64_t lda, const void *B, int64_t ldb, void *C,
                         int64_t ldc, int64_t M, int64_t N, int64_t K,
                         const qgemm_epilogue *epilogue, void *stream);
qgemm_status qgemm_w4a16_ex(const void *A_f16, int64_t lda, int64_t M, const qgemm_tensor *W,
                            void *C_f16, int64_t ldc, const qgemm_epilogue *epilogue,
                            void *stream);
qgemm_status qgemm_w4a16_f16s_ex(const void *A_f16, int64_t lda, int64_t M, const void *W_int4,
                                 int64_t ldw_bytes, const void *scales_f16, int64_t lds,
                                 int64_t N, int64_t K, void *C_f16, int64_t ldc,
                                 const qgemm_epilogue *epilogue, void *stream);
qgemm_status qgemm_w8_gemv_ex(const void *X_f16, int64_t ldx, int64_t M, const qgemm_tensor *W,
                              void *Y_f16, int64_t ldy, const qgemm_epilogue *epilogue,
                              void *stream);

/* Dequantise-only debug kernel: out[r, k] = decode(t.data[r, k]) * 2^(t.scales[r, k/32] - 127)
 * as fp32 (fp16 views: the value itself), written densely as [rows, k] row-major.  Exists so
 * that the decoded operand values can be compared bit for bit with the CPU reference, as the
 * "Running inline ML operations in a shader with Metal 4" sample checks its GPU result against a
 * CPU implementation.  E4M3 NaN codes and scale byte 255 give NaN (E2M1 has no NaN code).
 * Errors: INVALID_ARG (null t or out); CUDA. */
qgemm_status qgemm_dequant_debug(const qgemm_tensor *t, float *out, void *stream);

/* Human-readable name of a status code (static string, never NULL).
 * Passage: "Optimize custom machine learning operations with Metal tensors", section "Creating
 * quantized tensors with scale factors" (a failed creation hands back an error object the caller
 * can read) and "TileLang Metal Backend Internals", section 5.8 "Developer Checklist" (an
 * unsupported shape should produce a clear error). */
const char *qgemm_status_string(qgemm_status s);

/* Detail of the last error returned on the calling thread (static per-thread buffer). */
const char *qgemm_last_error_message(void);

/* Synchronise `stream`, then read and clear the device error word of the current device.
 * *code_out (may be NULL) receives the raw word: 0 = no kernel gave up; otherwise bits name the
 * wait that ran out (1 producer, 2 MMA issuer, 4 epilogue, 8 drain, 16 test wait) or, in the
 * debug build (libqgemm_debug.so, compiled with QGEMM_DEBUG), 32 = a kernel's own bounds check
 * failed and the access was skipped.
 * Returns QGEMM_ERR_TIMEOUT if the word was non-zero, QGEMM_ERR_CUDA if synchronisation failed. */
qgemm_status qgemm_poll_device_error(void *stream, uint32_t *code_out);

/* Upper bound, in nanoseconds, on every device-side wait of kernels launched after this call
 * (default 4e9).  Values below 1e6 are raised to 1e6. */
void qgemm_set_wait_timeout_ns(uint64_t ns);

/* Failure-detection self test: launches one kernel that waits on a barrier nothing ever
 * completes, with the wait limit `timeout_ns`; the wait gives up, records bit 16 in the device
 * error word and the kernel returns normally.  No output; use qgemm_poll_device_error().
 * Errors: CUDA. */
qgemm_status qgemm_selftest_wait_timeout(uint64_t timeout_ns, void *stream);

/* Measurement aid: the SM clock over a window of wall time, read on the GPU.  Launches one
 * 32-thread block that reads the SM cycle counter (clock64) and the global nanosecond timer, naps
 * until window_ns have passed on that timer, reads both again and writes out_dev[0] = cycles and
 * out_dev[1] = nanoseconds elapsed (device memory, two uint64); cycles / nanoseconds is the clock
 * in GHz.  The block is launched as a programmatic dependent of the kernel before it on `stream`:
 * issued right after a qgemm_mxfp8 / qgemm_mxfp4 call on the same stream, it starts once every CTA
 * of that GEMM runs, takes almost no room beside them, reports the clock the GEMM runs at (under a
 * power cap the SM clock drops below its maximum) and completes only after the GEMM has; give it
 * a window shorter than the GEMM.  After other work it simply runs next.
 * The pages have no counterpart: benchmarks of compute-bound kernels need the clock they ran at.
 * Errors: INVALID_ARG (out NULL, window 0 or above 1e9 ns), MISALIGNED (out not 8-byte
 * aligned); CUDA. */
qgemm_status qgemm_sm_clock_probe(uint64_t window_ns, uint64_t *out_dev, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* QGEMM_H */
