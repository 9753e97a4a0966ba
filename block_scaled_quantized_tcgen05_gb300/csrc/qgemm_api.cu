// qgemm_api.cu -- the C ABI: argument validation, tensor views, TMA descriptor encoding, the
// device error word and status strings.  Kernels live in the other translation units.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <atomic>
#include <mutex>
#include <new>

#include "qgemm.h"
#include "qgemm_internal.h"

namespace {

// Device error word: a kernel whose bounded wait ran out sets a bit here.  Host code reaches it
// only through the address returned by cudaGetSymbolAddress on the current device.
__device__ unsigned int g_device_error_word;

thread_local char g_last_msg[512] = "";

// bound on every device-side wait; set from any host thread, read at each launch
std::atomic<uint64_t> g_timeout_ns{4000000000ull};

constexpr int MAX_DEVICES = 64;
struct DeviceInfo {
    bool ready = false;
    int num_sms = 0;
    unsigned *err = nullptr;
    cudaMemPool_t pool = nullptr;   // scratch pool, created on first use
};
DeviceInfo g_dev[MAX_DEVICES];
std::mutex g_dev_mutex;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

qgemm_status cuda_fail(cudaError_t e, const char *what) {
    return qgi::fail(QGEMM_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e),
                     cudaGetErrorString(e));
}

// Per-device set-up on the current device: SM count and the address of the error word.
qgemm_status get_ctx(void *stream, qgi::LaunchCtx *ctx) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= MAX_DEVICES) return qgi::fail(QGEMM_ERR_CUDA, "device index %d", dev);
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_device_error_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
        d.err = static_cast<unsigned *>(p);
        d.ready = true;
    }
    ctx->stream = static_cast<cudaStream_t>(stream);
    ctx->err = d.err;
    ctx->timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
    ctx->num_sms = d.num_sms;
    ctx->device = dev;
    return QGEMM_OK;
}

}  // namespace

namespace qgi {

cudaError_t scratch_alloc(size_t bytes, const LaunchCtx &ctx, void **p) {
    cudaMemPool_t pool;
    {
        std::lock_guard<std::mutex> lock(g_dev_mutex);
        DeviceInfo &d = g_dev[ctx.device];
        if (!d.pool) {
            cudaMemPoolProps props = {};
            props.allocType = cudaMemAllocationTypePinned;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = ctx.device;
            cudaError_t e = cudaMemPoolCreate(&d.pool, &props);
            if (e != cudaSuccess) {
                d.pool = nullptr;
                return e;
            }
            uint64_t keep = UINT64_MAX;   // never hand memory back at synchronisation points
            e = cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep);
            if (e != cudaSuccess) return e;
        }
        pool = d.pool;
    }
    return cudaMallocFromPoolAsync(p, bytes, pool, ctx.stream);
}

cudaError_t scratch_free(void *p, const LaunchCtx &ctx) {
    return p ? cudaFreeAsync(p, ctx.stream) : cudaSuccess;
}

qgemm_status launch_ctx(void *stream, LaunchCtx *ctx) { return get_ctx(stream, ctx); }

}  // namespace qgi

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t elem_bits(int32_t dt) {
    switch (dt) {
    case QGEMM_F16: return 16;
    case QGEMM_E4M3:
    case QGEMM_INT8: return 8;
    case QGEMM_INT4:
    case QGEMM_E2M1: return 4;
    default: return 0;
    }
}

constexpr int64_t MAX_DIM = (int64_t(1) << 31) - 1;

}  // namespace

namespace qgi {

qgemm_status fail(qgemm_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_msg, sizeof(g_last_msg), fmt, ap);
    va_end(ap);
    return s;
}

// The driver's tensor-map encoder, looked up once; records an error and returns null if absent.
static EncodeTiledFn get_encode() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    if (!g_encode) fail(QGEMM_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    return g_encode;
}

bool encode_tma_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t inner,
                   uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                   uint32_t box_outer, CUtensorMapSwizzle swizzle) {
    if (!get_encode()) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        fail(QGEMM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d): dims %llu x %llu stride %llu",
             static_cast<int>(r), (unsigned long long)inner, (unsigned long long)outer,
             (unsigned long long)row_stride_bytes);
        return false;
    }
    return true;
}

bool encode_tma_3d(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t d0,
                   uint64_t d1, uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes,
                   uint32_t box0, uint32_t box1, uint32_t box2, CUtensorMapSwizzle swizzle) {
    if (!get_encode()) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    const cuuint32_t box[3] = {box0, box1, box2};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        fail(QGEMM_ERR_CUDA, "cuTensorMapEncodeTiled (3-D) failed (%d)", static_cast<int>(r));
        return false;
    }
    return true;
}

}  // namespace qgi

using qgi::fail;

extern "C" {

int32_t qgemm_version(void) { return (1 << 16) | 0; }

int32_t qgemm_debug_build(void) {
#ifdef QGEMM_DEBUG
    return 1;
#else
    return 0;
#endif
}

const char *qgemm_status_string(qgemm_status s) {
    switch (s) {
    case QGEMM_OK: return "QGEMM_OK";
    case QGEMM_ERR_INVALID_ARG: return "QGEMM_ERR_INVALID_ARG";
    case QGEMM_ERR_UNSUPPORTED_SHAPE: return "QGEMM_ERR_UNSUPPORTED_SHAPE";
    case QGEMM_ERR_MISALIGNED: return "QGEMM_ERR_MISALIGNED";
    case QGEMM_ERR_UNSUPPORTED_DTYPE: return "QGEMM_ERR_UNSUPPORTED_DTYPE";
    case QGEMM_ERR_CUDA: return "QGEMM_ERR_CUDA";
    case QGEMM_ERR_TIMEOUT: return "QGEMM_ERR_TIMEOUT";
    }
    return "QGEMM_ERR_UNKNOWN";
}

const char *qgemm_last_error_message(void) { return g_last_msg; }

void qgemm_set_wait_timeout_ns(uint64_t ns) {
    g_timeout_ns.store(ns < 1000000ull ? 1000000ull : ns, std::memory_order_relaxed);
}

qgemm_status qgemm_create_tensor(qgemm_tensor **out, qgemm_dtype dt, int64_t rows, int64_t k,
                                 const void *data, int64_t data_row_stride_bytes,
                                 const uint8_t *scales_ue8m0, int64_t scale_row_stride_bytes,
                                 int32_t block_k) {
    if (!out) return fail(QGEMM_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    const int64_t bits = elem_bits(dt);
    if (bits == 0) return fail(QGEMM_ERR_UNSUPPORTED_DTYPE, "unknown dtype %d", (int)dt);
    if (rows < 0 || k < 0) return fail(QGEMM_ERR_INVALID_ARG, "negative shape");
    if (rows > MAX_DIM || k > MAX_DIM) return fail(QGEMM_ERR_UNSUPPORTED_SHAPE, "dimension >= 2^31");
    if (!data && rows * k > 0) return fail(QGEMM_ERR_INVALID_ARG, "data is NULL");
    const int64_t row_bytes = (k * bits + 7) / 8;
    if (rows > 1 && data_row_stride_bytes < row_bytes)
        return fail(QGEMM_ERR_INVALID_ARG, "data row stride %lld < row size %lld",
                    (long long)data_row_stride_bytes, (long long)row_bytes);
    if (data_row_stride_bytes < 0) return fail(QGEMM_ERR_INVALID_ARG, "negative data stride");
    if (dt == QGEMM_F16) {
        if (scales_ue8m0) return fail(QGEMM_ERR_UNSUPPORTED_DTYPE, "F16 takes no scale plane");
    } else {
        if (block_k != 32)
            return fail(QGEMM_ERR_UNSUPPORTED_DTYPE, "block_k must be 32 (got %d)", block_k);
        if (k % 32) return fail(QGEMM_ERR_UNSUPPORTED_SHAPE, "k %% 32 != 0 (k = %lld)", (long long)k);
        if (!scales_ue8m0 && rows * k > 0) return fail(QGEMM_ERR_INVALID_ARG, "scales is NULL");
        if (scale_row_stride_bytes < 0 || (rows > 1 && scale_row_stride_bytes < k / 32))
            return fail(QGEMM_ERR_INVALID_ARG, "scale row stride %lld < k/32",
                        (long long)scale_row_stride_bytes);
    }
    qgemm_tensor *t = new (std::nothrow) qgemm_tensor;
    if (!t) return fail(QGEMM_ERR_INVALID_ARG, "out of host memory");
    t->dtype = dt;
    t->rows = rows;
    t->k = k;
    t->data = static_cast<const uint8_t *>(data);
    t->ld = data_row_stride_bytes;
    t->scales = scales_ue8m0;
    t->lds = scale_row_stride_bytes;
    *out = t;
    return QGEMM_OK;
}

qgemm_status qgemm_tensor_slice(const qgemm_tensor *t, int64_t row0, int64_t nrows, int64_t k0,
                                int64_t nk, qgemm_tensor **out) {
    if (!out) return fail(QGEMM_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!t) return fail(QGEMM_ERR_INVALID_ARG, "tensor is NULL");
    if (row0 < 0 || nrows < 0 || k0 < 0 || nk < 0 || row0 + nrows > t->rows || k0 + nk > t->k)
        return fail(QGEMM_ERR_INVALID_ARG, "slice out of range");
    if (t->dtype != QGEMM_F16 && (k0 % 32 || nk % 32))
        return fail(QGEMM_ERR_UNSUPPORTED_SHAPE, "k0 and nk must be multiples of 32");
    qgemm_tensor *s = new (std::nothrow) qgemm_tensor(*t);
    if (!s) return fail(QGEMM_ERR_INVALID_ARG, "out of host memory");
    const int64_t bits = elem_bits(t->dtype);
    s->rows = nrows;
    s->k = nk;
    s->data = t->data + row0 * t->ld + (k0 * bits) / 8;
    if (t->scales) s->scales = t->scales + row0 * t->lds + k0 / 32;
    *out = s;
    return QGEMM_OK;
}

void qgemm_destroy_tensor(qgemm_tensor *t) { delete t; }

qgemm_status qgemm_tensor_info(const qgemm_tensor *t, int32_t *dtype, int64_t *rows, int64_t *k,
                               const void **data, int64_t *data_row_stride_bytes,
                               const uint8_t **scales, int64_t *scale_row_stride_bytes) {
    if (!t) return fail(QGEMM_ERR_INVALID_ARG, "tensor is NULL");
    if (dtype) *dtype = t->dtype;
    if (rows) *rows = t->rows;
    if (k) *k = t->k;
    if (data) *data = t->data;
    if (data_row_stride_bytes) *data_row_stride_bytes = t->ld;
    if (scales) *scales = t->scales;
    if (scale_row_stride_bytes) *scale_row_stride_bytes = t->lds;
    return QGEMM_OK;
}

static qgemm_status check_out_f16(const void *C, int64_t ldc, int64_t M, int64_t N) {
    if (M * N == 0) return QGEMM_OK;
    if (!C) return fail(QGEMM_ERR_INVALID_ARG, "output is NULL");
    if (ldc < N) return fail(QGEMM_ERR_INVALID_ARG, "ldc %lld < N %lld", (long long)ldc, (long long)N);
    if (!aligned(C, 2)) return fail(QGEMM_ERR_MISALIGNED, "output must be 2-byte aligned");
    return QGEMM_OK;
}

static qgemm_status mxfp8_impl(const qgemm_tensor *A, const qgemm_tensor *B, void *C,
                               int64_t ldc, int epi, void *stream) {
    if (!A || !B) return fail(QGEMM_ERR_INVALID_ARG, "A or B is NULL");
    if (A->dtype != QGEMM_E4M3 || B->dtype != QGEMM_E4M3)
        return fail(QGEMM_ERR_UNSUPPORTED_DTYPE, "qgemm_mxfp8 takes E4M3 views");
    if (A->k != B->k) return fail(QGEMM_ERR_INVALID_ARG, "K mismatch (%lld vs %lld)",
                                  (long long)A->k, (long long)B->k);
    const int64_t M = A->rows, N = B->rows, K = A->k;
    qgemm_status st = check_out_f16(C, ldc, M, N);
    if (st != QGEMM_OK) return st;
    if (M == 0 || N == 0) return QGEMM_OK;
    if (K % 32) return fail(QGEMM_ERR_UNSUPPORTED_SHAPE, "K %% 32 != 0");
    for (const qgemm_tensor *t : {A, B}) {
        if (K > 0 && (!aligned(t->data, 16) || t->ld % 16))
            return fail(QGEMM_ERR_MISALIGNED, "E4M3 data must be 16-byte aligned, row stride %% 16 == 0");
    }
    qgi::LaunchCtx ctx;
    st = get_ctx(stream, &ctx);
    if (st != QGEMM_OK) return st;
    ctx.epi = epi;
    cudaError_t e;
    if (K == 0) {
        e = qgi::launch_empty_sum_epilogue(static_cast<__half *>(C), ldc, M, N, ctx);
        return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "empty-sum epilogue");
    }
    bool enc = true;
    e = qgi::launch_mxfp8(A, B, static_cast<__half *>(C), ldc, ctx, &enc);
    if (!enc) return QGEMM_ERR_CUDA;
    return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "qgemm_mxfp8 launch");
}

static qgemm_status mxfp4_impl(const qgemm_tensor *A, const qgemm_tensor *B, void *C,
                               int64_t ldc, int epi, void *stream) {
    if (!A || !B) return fail(QGEMM_ERR_INVALID_ARG, "A or B is NULL");
    if (A->dtype != QGEMM_E2M1 || B->dtype != QGEMM_E2M1)
        return fail(QGEMM_ERR_UNSUPPORTED_DTYPE, "qgemm_mxfp4 takes E2M1 views");
    if (A->k != B->k) return fail(QGEMM_ERR_INVALID_ARG, "K mismatch (%lld vs %lld)",
                                  (long long)A->k, (long long)B->k);
    const int64_t M = A->rows, N = B->rows, K = A->k;
    qgemm_status st = check_out_f16(C, ldc, M, N);
    if (st != QGEMM_OK) return st;
    if (M == 0 || N == 0) return QGEMM_OK;
    if (K % 32) return fail(QGEMM_ERR_UNSUPPORTED_SHAPE, "K %% 32 != 0");
    for (const qgemm_tensor *t : {A, B}) {
        if (K > 0 && (!aligned(t->data, 16) || t->ld % 16))
            return fail(QGEMM_ERR_MISALIGNED, "E2M1 data must be 16-byte aligned, row stride %% 16 == 0");
    }
    qgi::LaunchCtx ctx;
    st = get_ctx(stream, &ctx);
    if (st != QGEMM_OK) return st;
    ctx.epi = epi;
    cudaError_t e;
    if (K == 0) {
        e = qgi::launch_empty_sum_epilogue(static_cast<__half *>(C), ldc, M, N, ctx);
        return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "empty-sum epilogue");
    }
    void *scratch = nullptr;
    e = qgi::scratch_alloc(qgi::mxfp4_scratch_bytes(A, B), ctx, &scratch);
    if (e != cudaSuccess) return cuda_fail(e, "qgemm_mxfp4 scratch");
    bool enc = true;
    e = qgi::launch_mxfp4_pair(A, B, static_cast<__half *>(C), ldc, scratch, ctx, &enc);
    const cudaError_t f = qgi::scratch_free(scratch, ctx);
    if (!enc) return QGEMM_ERR_CUDA;
    if (e == cudaSuccess) e = f;
    return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "qgemm_mxfp4 launch");
}

static qgemm_status gemm_f16_impl(const void *A, int64_t lda, const void *B, int64_t ldb, void *C,
                                  int64_t ldc, int64_t M, int64_t N, int64_t K, int epi,
                                  void *stream) {
    if (M < 0 || N < 0 || K < 0) return fail(QGEMM_ERR_INVALID_ARG, "negative shape");
    if (M > MAX_DIM || N > MAX_DIM || K > MAX_DIM)
        return fail(QGEMM_ERR_UNSUPPORTED_SHAPE, "dimension >= 2^31");
    qgemm_status st = check_out_f16(C, ldc, M, N);
    if (st != QGEMM_OK) return st;
    if (M == 0 || N == 0) return QGEMM_OK;
    if (K > 0) {
        if (!A || !B) return fail(QGEMM_ERR_INVALID_ARG, "A or B is NULL");
        if (lda < K || ldb < N) return fail(QGEMM_ERR_INVALID_ARG, "lda < K or ldb < N");
        if (!aligned(A, 16) || !aligned(B, 16) || lda % 8 || ldb % 8)
            return fail(QGEMM_ERR_MISALIGNED, "A, B must be 16-byte aligned, lda/ldb %% 8 == 0");
    }
    qgi::LaunchCtx ctx;
    st = get_ctx(stream, &ctx);
    if (st != QGEMM_OK) return st;
    ctx.epi = epi;
    cudaError_t e;
    if (K == 0) {
        e = qgi::launch_empty_sum_epilogue(static_cast<__half *>(C), ldc, M, N, ctx);
        return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "empty-sum epilogue");
    }
    bool enc = true;
    e = qgi::launch_gemm_f16(static_cast<const __half *>(A), lda, static_cast<const __half *>(B),
                             ldb, static_cast<__half *>(C), ldc, (int)M, (int)N, (int)K, ctx, &enc);
    if (!enc) return QGEMM_ERR_CUDA;
    return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "gemm_f16 launch");
}

static qgemm_status w4a16_impl(const void *A_f16, int64_t lda, int64_t M, const qgemm_tensor *W,
                               void *C_f16, int64_t ldc, int epi, void *stream) {
    if (!W) return fail(QGEMM_ERR_INVALID_ARG, "W is NULL");
    if (W->dtype != QGEMM_INT4) return fail(QGEMM_ERR_UNSUPPORTED_DTYPE, "W must be an INT4 view");
    if (M < 0) return fail(QGEMM_ERR_INVALID_ARG, "negative M");
    if (M > MAX_DIM) return fail(QGEMM_ERR_UNSUPPORTED_SHAPE, "M >= 2^31");
    const int64_t N = W->rows, K = W->k;
    qgemm_status st = check_out_f16(C_f16, ldc, M, N);
    if (st != QGEMM_OK) return st;
    if (M == 0 || N == 0) return QGEMM_OK;
    if (K % 64) return fail(QGEMM_ERR_UNSUPPORTED_SHAPE, "K %% 64 != 0 (K = %lld)", (long long)K);
    if (K > 0) {
        if (!A_f16) return fail(QGEMM_ERR_INVALID_ARG, "A is NULL");
        if (lda < K) return fail(QGEMM_ERR_INVALID_ARG, "lda < K");
        if (!aligned(A_f16, 16) || lda % 8)
            return fail(QGEMM_ERR_MISALIGNED, "A must be 16-byte aligned, lda %% 8 == 0");
        if (!aligned(W->data, 16) || W->ld % 16)
            return fail(QGEMM_ERR_MISALIGNED, "int4 data must be 16-byte aligned, stride %% 16 == 0");
    }
    qgi::LaunchCtx ctx;
    st = get_ctx(stream, &ctx);
    if (st != QGEMM_OK) return st;
    ctx.epi = epi;
    cudaError_t e;
    if (K == 0) {
        e = qgi::launch_empty_sum_epilogue(static_cast<__half *>(C_f16), ldc, M, N, ctx);
        return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "empty-sum epilogue");
    }
    bool enc = true;
    e = qgi::launch_w4a16(static_cast<const __half *>(A_f16), lda, (int)M, W,
                          static_cast<__half *>(C_f16), ldc, ctx, &enc);
    if (!enc) return QGEMM_ERR_CUDA;
    if (e != cudaSuccess) return cuda_fail(e, "qgemm_w4a16 launch");
    // rows with nonzero weights under scale bytes outside the fold window, from the definition
    e = qgi::launch_w4a16_outliers(static_cast<const __half *>(A_f16), lda, (int)M, W,
                                   static_cast<__half *>(C_f16), ldc, ctx);
    return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "qgemm_w4a16 outlier-row launch");
}

static qgemm_status w4a16_f16s_impl(const void *A_f16, int64_t lda, int64_t M, const void *W_int4,
                                    int64_t ldw, const void *scales_f16, int64_t lds, int64_t N,
                                    int64_t K, void *C_f16, int64_t ldc, int epi, void *stream) {
    if (M < 0 || N < 0 || K < 0) return fail(QGEMM_ERR_INVALID_ARG, "negative shape");
    if (M > MAX_DIM || N > MAX_DIM || K > MAX_DIM)
        return fail(QGEMM_ERR_UNSUPPORTED_SHAPE, "dimension >= 2^31");
    qgemm_status st = check_out_f16(C_f16, ldc, M, N);
    if (st != QGEMM_OK) return st;
    if (M == 0 || N == 0) return QGEMM_OK;
    if (K % 256) return fail(QGEMM_ERR_UNSUPPORTED_SHAPE, "K %% 256 != 0 (K = %lld)", (long long)K);
    if (K > 0) {
        if (!A_f16 || !W_int4 || !scales_f16)
            return fail(QGEMM_ERR_INVALID_ARG, "A, W or scales is NULL");
        if (lda < K || ldw < K / 2 || lds < K / 32)
            return fail(QGEMM_ERR_INVALID_ARG, "lda < K, ldw < K/2 bytes or lds < K/32");
        if (!aligned(A_f16, 16) || lda % 8)
            return fail(QGEMM_ERR_MISALIGNED, "A must be 16-byte aligned, lda %% 8 == 0");
        if (!aligned(W_int4, 16) || ldw % 16)
            return fail(QGEMM_ERR_MISALIGNED, "int4 data must be 16-byte aligned, stride %% 16 == 0");
        if (!aligned(scales_f16, 16) || lds % 8)
            return fail(QGEMM_ERR_MISALIGNED, "fp16 scales must be 16-byte aligned, lds %% 8 == 0");
    }
    qgi::LaunchCtx ctx;
    st = get_ctx(stream, &ctx);
    if (st != QGEMM_OK) return st;
    ctx.epi = epi;
    cudaError_t e;
    if (K == 0) {
        e = qgi::launch_empty_sum_epilogue(static_cast<__half *>(C_f16), ldc, M, N, ctx);
        return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "empty-sum epilogue");
    }
    bool enc = true;
    e = qgi::launch_w4a16_f16s(static_cast<const __half *>(A_f16), lda, (int)M,
                               static_cast<const uint8_t *>(W_int4), ldw,
                               static_cast<const __half *>(scales_f16), lds, (int)N, (int)K,
                               static_cast<__half *>(C_f16), ldc, ctx, &enc);
    if (!enc) return QGEMM_ERR_CUDA;
    return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "qgemm_w4a16_f16s launch");
}

static qgemm_status w8_gemv_impl(const void *X_f16, int64_t ldx, int64_t M, const qgemm_tensor *W,
                                 void *Y_f16, int64_t ldy, int epi, void *stream) {
    if (!W) return fail(QGEMM_ERR_INVALID_ARG, "W is NULL");
    if (W->dtype != QGEMM_INT8) return fail(QGEMM_ERR_UNSUPPORTED_DTYPE, "W must be an INT8 view");
    if (M < 1 || M > 16) return fail(QGEMM_ERR_UNSUPPORTED_SHAPE, "M must be in 1..16 (got %lld)",
                                     (long long)M);
    const int64_t N = W->rows, K = W->k;
    if (N == 0) return QGEMM_OK;
    if (!Y_f16) return fail(QGEMM_ERR_INVALID_ARG, "Y is NULL");
    if (ldy < N) return fail(QGEMM_ERR_INVALID_ARG, "ldy < N");
    if (!aligned(Y_f16, 2)) return fail(QGEMM_ERR_MISALIGNED, "Y must be 2-byte aligned");
    if (K % 32) return fail(QGEMM_ERR_UNSUPPORTED_SHAPE, "K %% 32 != 0");
    if (K > 0) {
        if (!X_f16) return fail(QGEMM_ERR_INVALID_ARG, "X is NULL");
        if (ldx < K) return fail(QGEMM_ERR_INVALID_ARG, "ldx < K");
        if (!aligned(X_f16, 16) || ldx % 8)
            return fail(QGEMM_ERR_MISALIGNED, "X must be 16-byte aligned, ldx %% 8 == 0");
        if (!aligned(W->data, 16) || W->ld % 16)
            return fail(QGEMM_ERR_MISALIGNED, "int8 data must be 16-byte aligned, stride %% 16 == 0");
    }
    qgi::LaunchCtx ctx;
    qgemm_status st = get_ctx(stream, &ctx);
    if (st != QGEMM_OK) return st;
    ctx.epi = epi;
    cudaError_t e;
    if (K == 0) {
        e = qgi::launch_empty_sum_epilogue(static_cast<__half *>(Y_f16), ldy, M, N, ctx);
        return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "empty-sum epilogue");
    }
    bool enc = true;
    e = qgi::launch_w8_gemv(static_cast<const __half *>(X_f16), ldx, (int)M, W,
                            static_cast<__half *>(Y_f16), ldy, ctx, &enc);
    if (!enc) return QGEMM_ERR_CUDA;
    return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "qgemm_w8_gemv launch");
}

// Epilogue descriptor -> EPI_* flags (NULL: plain store).
static qgemm_status epi_flags(const qgemm_epilogue *ep, int *flags) {
    *flags = 0;
    if (!ep) return QGEMM_OK;
    if ((ep->accumulate != 0 && ep->accumulate != 1) || (ep->relu != 0 && ep->relu != 1))
        return fail(QGEMM_ERR_INVALID_ARG, "epilogue fields must be 0 or 1 (accumulate %d, relu %d)",
                    ep->accumulate, ep->relu);
    *flags = (ep->accumulate ? qgi::EPI_ACCUMULATE : 0) | (ep->relu ? qgi::EPI_RELU : 0);
    return QGEMM_OK;
}

qgemm_status qgemm_mxfp8(const qgemm_tensor *A, const qgemm_tensor *B, void *C, int64_t ldc,
                         void *stream) {
    return mxfp8_impl(A, B, C, ldc, 0, stream);
}

qgemm_status qgemm_mxfp8_ex(const qgemm_tensor *A, const qgemm_tensor *B, void *C, int64_t ldc,
                            const qgemm_epilogue *epilogue, void *stream) {
    int f;
    const qgemm_status st = epi_flags(epilogue, &f);
    return st != QGEMM_OK ? st : mxfp8_impl(A, B, C, ldc, f, stream);
}

qgemm_status qgemm_mxfp8_scratch_bytes(const qgemm_tensor *A, const qgemm_tensor *B,
                                       int64_t *bytes) {
    if (!bytes) return fail(QGEMM_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = 0;
    if (!A || !B) return fail(QGEMM_ERR_INVALID_ARG, "A or B is NULL");
    if (A->dtype != QGEMM_E4M3 || B->dtype != QGEMM_E4M3)
        return fail(QGEMM_ERR_UNSUPPORTED_DTYPE, "qgemm_mxfp8 takes E4M3 views");
    if (A->k != B->k) return fail(QGEMM_ERR_INVALID_ARG, "K mismatch (%lld vs %lld)",
                                  (long long)A->k, (long long)B->k);
    qgi::LaunchCtx ctx;
    const qgemm_status st = get_ctx(nullptr, &ctx);
    if (st != QGEMM_OK) return st;
    *bytes = static_cast<int64_t>(qgi::mxfp8_scratch_bytes(A, B, ctx.num_sms));
    return QGEMM_OK;
}

qgemm_status qgemm_mxfp4(const qgemm_tensor *A, const qgemm_tensor *B, void *C, int64_t ldc,
                         void *stream) {
    return mxfp4_impl(A, B, C, ldc, 0, stream);
}

qgemm_status qgemm_mxfp4_ex(const qgemm_tensor *A, const qgemm_tensor *B, void *C, int64_t ldc,
                            const qgemm_epilogue *epilogue, void *stream) {
    int f;
    const qgemm_status st = epi_flags(epilogue, &f);
    return st != QGEMM_OK ? st : mxfp4_impl(A, B, C, ldc, f, stream);
}

qgemm_status gemm_f16(const void *A, int64_t lda, const void *B, int64_t ldb, void *C,
                      int64_t ldc, int64_t M, int64_t N, int64_t K, void *stream) {
    return gemm_f16_impl(A, lda, B, ldb, C, ldc, M, N, K, 0, stream);
}

qgemm_status gemm_f16_ex(const void *A, int64_t lda, const void *B, int64_t ldb, void *C,
                         int64_t ldc, int64_t M, int64_t N, int64_t K,
                         const qgemm_epilogue *epilogue, void *stream) {
    int f;
    const qgemm_status st = epi_flags(epilogue, &f);
    return st != QGEMM_OK ? st : gemm_f16_impl(A, lda, B, ldb, C, ldc, M, N, K, f, stream);
}

qgemm_status qgemm_w4a16(const void *A_f16, int64_t lda, int64_t M, const qgemm_tensor *W,
                         void *C_f16, int64_t ldc, void *stream) {
    return w4a16_impl(A_f16, lda, M, W, C_f16, ldc, 0, stream);
}

qgemm_status qgemm_w4a16_ex(const void *A_f16, int64_t lda, int64_t M, const qgemm_tensor *W,
                            void *C_f16, int64_t ldc, const qgemm_epilogue *epilogue,
                            void *stream) {
    int f;
    const qgemm_status st = epi_flags(epilogue, &f);
    return st != QGEMM_OK ? st : w4a16_impl(A_f16, lda, M, W, C_f16, ldc, f, stream);
}

qgemm_status qgemm_attention_f16(const void *Q, const void *K, const void *V, void *O, int64_t BH,
                                 int64_t Lq, int64_t Lk, int64_t d, int64_t q_head_stride,
                                 int64_t q_row_stride, int64_t k_head_stride, int64_t k_row_stride,
                                 int64_t v_head_stride, int64_t v_row_stride,
                                 int64_t o_head_stride, int64_t o_row_stride, float scale,
                                 void *stream) {
    if (BH < 0 || Lq < 0 || Lk < 0 || d < 0) return fail(QGEMM_ERR_INVALID_ARG, "negative shape");
    if (BH == 0 || Lq == 0) return QGEMM_OK;
    if (d != 128) return fail(QGEMM_ERR_UNSUPPORTED_SHAPE, "head dimension must be 128 (got %lld)",
                              (long long)d);
    if (Lk == 0) return fail(QGEMM_ERR_UNSUPPORTED_SHAPE, "Lk = 0: softmax over no keys");
    if (BH > 65535 || Lq > MAX_DIM || Lk > MAX_DIM)
        return fail(QGEMM_ERR_UNSUPPORTED_SHAPE, "BH > 65535 or a length >= 2^31");
    if (!(scale > 0.0f) || !isfinite(scale))
        return fail(QGEMM_ERR_INVALID_ARG, "scale must be finite and > 0");
    if (!Q || !K || !V || !O) return fail(QGEMM_ERR_INVALID_ARG, "Q, K, V or O is NULL");
    struct View { const void *p; int64_t hs, rs, L; const char *name; };
    const View views[4] = {{Q, q_head_stride, q_row_stride, Lq, "Q"},
                           {K, k_head_stride, k_row_stride, Lk, "K"},
                           {V, v_head_stride, v_row_stride, Lk, "V"},
                           {O, o_head_stride, o_row_stride, Lq, "O"}};
    for (const View &v : views) {
        if (v.rs < 0 || v.hs < 0) return fail(QGEMM_ERR_INVALID_ARG, "%s: negative stride", v.name);
        if (!aligned(v.p, 16) || v.rs % 8 || v.hs % 8)
            return fail(QGEMM_ERR_MISALIGNED, "%s must be 16-byte aligned with strides %% 8 == 0",
                        v.name);
    }
    // O's rows must not overlap: heads outside rows ([BH, Lq, d]) or rows outside heads
    // ([Lq, BH, d], e.g. a [batch, L, heads, d] buffer)
    const bool heads_outer = (BH == 1 || o_head_stride >= Lq * o_row_stride) && o_row_stride >= d;
    const bool rows_outer = (Lq == 1 || o_row_stride >= BH * o_head_stride) && o_head_stride >= d;
    if (!heads_outer && !rows_outer)
        return fail(QGEMM_ERR_INVALID_ARG, "O strides make output rows overlap");
    qgi::LaunchCtx ctx;
    qgemm_status st = get_ctx(stream, &ctx);
    if (st != QGEMM_OK) return st;
    qgi::AttnArgs a;
    a.Q = static_cast<const __half *>(Q);
    a.K = static_cast<const __half *>(K);
    a.V = static_cast<const __half *>(V);
    a.O = static_cast<__half *>(O);
    // a stride that is never stepped (one head, one row) may be anything; the tensor maps need a
    // positive multiple of 16 bytes there
    auto eff = [](int64_t stride, int64_t extent) { return extent > 1 || stride > 0 ? stride : 8; };
    a.q_hs = eff(q_head_stride, BH);
    a.k_hs = eff(k_head_stride, BH);
    a.v_hs = eff(v_head_stride, BH);
    a.o_hs = eff(o_head_stride, BH);
    a.q_rs = eff(q_row_stride, Lq);
    a.k_rs = eff(k_row_stride, Lk);
    a.v_rs = eff(v_row_stride, Lk);
    a.o_rs = eff(o_row_stride, Lq);
    a.BH = (int)BH;
    a.Lq = (int)Lq;
    a.Lk = (int)Lk;
    a.scale = scale;
    bool enc = true;
    const cudaError_t e = qgi::launch_attention(a, ctx, &enc);
    if (!enc) return QGEMM_ERR_CUDA;
    return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "qgemm_attention_f16 launch");
}

qgemm_status qgemm_w4a16_f16s(const void *A_f16, int64_t lda, int64_t M, const void *W_int4,
                              int64_t ldw_bytes, const void *scales_f16, int64_t lds, int64_t N,
                              int64_t K, void *C_f16, int64_t ldc, void *stream) {
    return w4a16_f16s_impl(A_f16, lda, M, W_int4, ldw_bytes, scales_f16, lds, N, K, C_f16, ldc, 0,
                           stream);
}

qgemm_status qgemm_w4a16_f16s_ex(const void *A_f16, int64_t lda, int64_t M, const void *W_int4,
                                 int64_t ldw_bytes, const void *scales_f16, int64_t lds,
                                 int64_t N, int64_t K, void *C_f16, int64_t ldc,
                                 const qgemm_epilogue *epilogue, void *stream) {
    int f;
    const qgemm_status st = epi_flags(epilogue, &f);
    return st != QGEMM_OK ? st
                          : w4a16_f16s_impl(A_f16, lda, M, W_int4, ldw_bytes, scales_f16, lds, N,
                                            K, C_f16, ldc, f, stream);
}

qgemm_status qgemm_w8_gemv(const void *X_f16, int64_t ldx, int64_t M, const qgemm_tensor *W,
                           void *Y_f16, int64_t ldy, void *stream) {
    return w8_gemv_impl(X_f16, ldx, M, W, Y_f16, ldy, 0, stream);
}

qgemm_status qgemm_w8_gemv_ex(const void *X_f16, int64_t ldx, int64_t M, const qgemm_tensor *W,
                              void *Y_f16, int64_t ldy, const qgemm_epilogue *epilogue,
                              void *stream) {
    int f;
    const qgemm_status st = epi_flags(epilogue, &f);
    return st != QGEMM_OK ? st : w8_gemv_impl(X_f16, ldx, M, W, Y_f16, ldy, f, stream);
}

qgemm_status qgemm_dequant_debug(const qgemm_tensor *t, float *out, void *stream) {
    if (!t) return fail(QGEMM_ERR_INVALID_ARG, "tensor is NULL");
    if (t->rows * t->k == 0) return QGEMM_OK;
    if (!out) return fail(QGEMM_ERR_INVALID_ARG, "out is NULL");
    qgi::LaunchCtx ctx;
    qgemm_status st = get_ctx(stream, &ctx);
    if (st != QGEMM_OK) return st;
    cudaError_t e = qgi::launch_dequant(t, out, ctx);
    return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "qgemm_dequant_debug launch");
}

qgemm_status qgemm_poll_device_error(void *stream, uint32_t *code_out) {
    if (code_out) *code_out = 0;
    qgi::LaunchCtx ctx;
    qgemm_status st = get_ctx(stream, &ctx);
    if (st != QGEMM_OK) return st;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned word = 0;
    e = cudaMemcpy(&word, ctx.err, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read device error word");
    if (word) {
        const unsigned zero = 0;
        e = cudaMemcpy(ctx.err, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
    }
    if (code_out) *code_out = word;
    if (word) return fail(QGEMM_ERR_TIMEOUT, "device error word 0x%x", word);
    return QGEMM_OK;
}

qgemm_status qgemm_sm_clock_probe(uint64_t window_ns, uint64_t *out_dev, void *stream) {
    if (!out_dev) return fail(QGEMM_ERR_INVALID_ARG, "out is NULL");
    if (window_ns == 0 || window_ns > 1000000000ull)
        return fail(QGEMM_ERR_INVALID_ARG, "window must be in 1 .. 1e9 ns (got %llu)",
                    (unsigned long long)window_ns);
    if (!aligned(out_dev, 8)) return fail(QGEMM_ERR_MISALIGNED, "out must be 8-byte aligned");
    qgi::LaunchCtx ctx;
    qgemm_status st = get_ctx(stream, &ctx);
    if (st != QGEMM_OK) return st;
    cudaError_t e = qgi::launch_clock_probe(window_ns, out_dev, ctx);
    return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "clock probe launch");
}

qgemm_status qgemm_selftest_wait_timeout(uint64_t timeout_ns, void *stream) {
    qgi::LaunchCtx ctx;
    qgemm_status st = get_ctx(stream, &ctx);
    if (st != QGEMM_OK) return st;
    cudaError_t e = qgi::launch_selftest_wait(timeout_ns, ctx);
    return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "self-test launch");
}

}  // extern "C"
