// mxfp8_noalloc.cu -- qgemm_mxfp8_noalloc: the MXFP8 GEMM without any device allocation.
//
// qgemm_mxfp8 takes a few megabytes of stream-ordered scratch from a library pool on every call
// that runs on CTA pairs (the scale planes rewritten into tensor-core order).  Some callers cannot
// let a library allocate device memory while they run: a serving process that reserves all device
// memory up front for its own allocator, or a latency-critical path that cannot risk an
// allocation that blocks or fails in the middle of a request.  This entry point runs the same
// kernels with the scratch in a fixed device array that is part of the library's image, so a call
// makes no cudaMalloc, no pool allocation and no allocating library call.
//
// The array's price and its rules:
//  * every GPU on which the array has been placed (see below) holds NOALLOC_SCRATCH_BYTES for it
//    until exit;
//  * a shape whose repacked scales need more than that is rejected (QGEMM_ERR_UNSUPPORTED_SHAPE),
//    nothing is launched;
//  * all calls on one device share the array: calls that overlap on the GPU (different streams
//    without ordering between them) race on it and give wrong results -- order them on one stream
//    or synchronise between them;
//  * the array keeps whatever the previous call left in it; nothing has to start at zero, because
//    the repack kernel rewrites every byte the GEMM then reads;
//  * host code cannot use the array's name as a device address (it names a host-side stand-in), so
//    the first call on each device looks the address up with cudaGetSymbolAddress, with that
//    device current, and caches it; that first call should come before any stream capture;
//  * the array lives in this file's own module, which CUDA loads lazily by default: the driver
//    places the 8 MiB in device memory at that first lookup, not when the library is loaded, so a
//    caller that reserves the rest of device memory for itself makes one call on each device
//    before it does (with CUDA_MODULE_LOADING=EAGER the array is placed when the context is made);
//  * the cached address belongs to the device's current context: after cudaDeviceReset (or any
//    teardown of the primary context) the library must not be used again in this process.
#include <cuda_runtime.h>

#include <mutex>

#include "qgemm.h"
#include "qgemm_internal.h"

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(8) << 20;   // 8 MiB, e.g. M = N = 16384, K = 8192

constexpr int MAX_DEVICES = 64;
void *g_scratch_addr[MAX_DEVICES];   // device address of the array, per device (set-up once)
std::mutex g_scratch_mutex;

}  // namespace

// The scratch itself: one copy in the memory of every device that loads this library.
static __device__ __align__(256) uint8_t g_mxfp8_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of the array on the current device `dev`; looked up on the first call only.
qgemm_status scratch_address(int dev, void **out) {
    if (dev < 0 || dev >= MAX_DEVICES) return qgi::fail(QGEMM_ERR_CUDA, "device index %d", dev);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_mxfp8_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return qgi::fail(QGEMM_ERR_CUDA, "cudaGetSymbolAddress(no-alloc scratch): %s (%s)",
                             cudaGetErrorName(e), cudaGetErrorString(e));
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return QGEMM_OK;
}

bool aligned_to(const void *p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

}  // namespace

extern "C" qgemm_status qgemm_mxfp8_noalloc(const qgemm_tensor *A, const qgemm_tensor *B,
                                            void *C, int64_t ldc, void *stream) {
    using qgi::fail;
    if (!A || !B) return fail(QGEMM_ERR_INVALID_ARG, "A or B is NULL");
    if (A->dtype != QGEMM_E4M3 || B->dtype != QGEMM_E4M3)
        return fail(QGEMM_ERR_UNSUPPORTED_DTYPE, "qgemm_mxfp8_noalloc takes E4M3 views");
    if (A->k != B->k)
        return fail(QGEMM_ERR_INVALID_ARG, "K mismatch (%lld vs %lld)", (long long)A->k,
                    (long long)B->k);
    const int64_t M = A->rows, N = B->rows, K = A->k;
    if (M * N > 0) {
        if (!C) return fail(QGEMM_ERR_INVALID_ARG, "output is NULL");
        if (ldc < N) return fail(QGEMM_ERR_INVALID_ARG, "ldc %lld < N %lld", (long long)ldc, (long long)N);
        if (!aligned_to(C, 2)) return fail(QGEMM_ERR_MISALIGNED, "output must be 2-byte aligned");
    }
    if (M == 0 || N == 0) return QGEMM_OK;
    if (K % 32) return fail(QGEMM_ERR_UNSUPPORTED_SHAPE, "K %% 32 != 0");
    for (const qgemm_tensor *t : {A, B})
        if (K > 0 && (!aligned_to(t->data, 16) || t->ld % 16))
            return fail(QGEMM_ERR_MISALIGNED, "E4M3 data must be 16-byte aligned, row stride %% 16 == 0");
    const bool pair = K > 0 && qgi::mxfp8_pair_eligible(A, B);
    if (pair) {
        const size_t need = qgi::mxfp8_pair_scratch_bytes(A, B);
        if (need > NOALLOC_SCRATCH_BYTES)
            return fail(QGEMM_ERR_UNSUPPORTED_SHAPE,
                        "qgemm_mxfp8_noalloc: M = %lld, N = %lld, K = %lld needs %zu bytes of "
                        "scale scratch, the library's fixed buffer holds %zu; use qgemm_mxfp8",
                        (long long)M, (long long)N, (long long)K, need, NOALLOC_SCRATCH_BYTES);
    }
    qgi::LaunchCtx ctx;
    qgemm_status st = qgi::launch_ctx(stream, &ctx);
    if (st != QGEMM_OK) return st;
    cudaError_t e;
    bool enc = true;
    if (K == 0) {
        e = qgi::launch_fill_zero_f16(static_cast<__half *>(C), ldc, M, N, ctx);
    } else if (pair) {
        void *scratch = nullptr;
        st = scratch_address(ctx.device, &scratch);
        if (st != QGEMM_OK) return st;
        e = qgi::launch_mxfp8_pair(A, B, static_cast<__half *>(C), ldc, scratch, ctx, &enc);
    } else {
        // one CTA per tile, K not split: this path uses no scratch
        e = qgi::launch_mxfp8(A, B, static_cast<__half *>(C), ldc, ctx, &enc, false);
    }
    if (!enc) return QGEMM_ERR_CUDA;
    if (e != cudaSuccess)
        return fail(QGEMM_ERR_CUDA, "qgemm_mxfp8_noalloc launch: %s (%s)", cudaGetErrorName(e),
                    cudaGetErrorString(e));
    return QGEMM_OK;
}
