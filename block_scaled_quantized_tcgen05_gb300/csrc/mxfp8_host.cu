// mxfp8_host.cu -- qgemm_mxfp8_host: the MXFP8 GEMM on operands and output in host memory.
//
// The call copies both operands (data and scale planes) to the device, runs the CTA-pair GEMM
// and copies C back, and overlaps the three: B goes first, then A in row chunks on an internal
// upload stream; the GEMM of each row chunk starts on the caller's stream as soon as that chunk
// has landed, and each finished chunk of C goes back on an internal download stream while the
// next chunk computes.  Host <-> device transfers are the bound of this call (the product takes
// about a third of the time of its copies at 8192^3), so the library keeps two sets of device
// buffers and alternates them between calls: the uploads of one call run while the previous
// call's downloads still occupy the other direction of the link.
//
// Device memory: the two buffer sets grow to the largest shape seen and stay allocated (per
// device) until the process exits; the repacked scale planes (B's once per call, then one row
// chunk of A's at a time) come from the library's stream-ordered pool, as for qgemm_mxfp8.
#include <cstdio>
#include <mutex>

#include "qgemm_internal.h"

namespace {

constexpr int MAX_DEV = 64;
constexpr int CHUNKS = 4;          // row chunks of A and C per call

struct HostSet {
    uint8_t *base = nullptr;
    size_t bytes = 0;
    cudaEvent_t free_ev = nullptr;   // recorded after the last download that read this set
    bool used = false;
};

struct HostCtx {
    std::mutex mu;
    bool ready = false;
    cudaStream_t up = nullptr, down = nullptr;
    cudaEvent_t ev_b = nullptr, ev_out = nullptr, ev_start = nullptr;
    cudaEvent_t ev_a[CHUNKS] = {}, ev_c[CHUNKS] = {};
    HostSet set[2];
    unsigned calls = 0;
};
HostCtx g_host[MAX_DEV];

qgemm_status cuda_err(cudaError_t e, const char *what) {
    return qgi::fail(QGEMM_ERR_CUDA, "qgemm_mxfp8_host: %s: %s", what, cudaGetErrorString(e));
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" qgemm_status qgemm_mxfp8_host(const qgemm_tensor *A, const qgemm_tensor *B, void *C,
                                         int64_t ldc, void *stream_) {
    if (!A || !B) return qgi::fail(QGEMM_ERR_INVALID_ARG, "A or B is NULL");
    if (A->dtype != QGEMM_E4M3 || B->dtype != QGEMM_E4M3)
        return qgi::fail(QGEMM_ERR_UNSUPPORTED_DTYPE, "qgemm_mxfp8_host takes E4M3 views");
    if (A->k != B->k)
        return qgi::fail(QGEMM_ERR_INVALID_ARG, "K mismatch (%lld vs %lld)", (long long)A->k,
                         (long long)B->k);
    const int64_t M = A->rows, N = B->rows, K = A->k;
    if (M == 0 || N == 0) return QGEMM_OK;
    if (!C) return qgi::fail(QGEMM_ERR_INVALID_ARG, "output is NULL");
    if (ldc < N) return qgi::fail(QGEMM_ERR_INVALID_ARG, "ldc %lld < N %lld", (long long)ldc,
                                  (long long)N);
    if (K % 32) return qgi::fail(QGEMM_ERR_UNSUPPORTED_SHAPE, "K %% 32 != 0");

    qgi::LaunchCtx ctx;
    qgemm_status st = qgi::launch_ctx(stream_, &ctx);
    if (st != QGEMM_OK) return st;
    if (ctx.device < 0 || ctx.device >= MAX_DEV)
        return qgi::fail(QGEMM_ERR_CUDA, "device index %d", ctx.device);
    HostCtx &h = g_host[ctx.device];
    std::lock_guard<std::mutex> lock(h.mu);
    cudaError_t e;
    if (!h.ready) {
        if ((e = cudaStreamCreateWithFlags(&h.up, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&h.down, cudaStreamNonBlocking)) != cudaSuccess)
            return cuda_err(e, "stream creation");
        cudaEvent_t *evs[] = {&h.ev_b, &h.ev_out, &h.ev_start, &h.set[0].free_ev, &h.set[1].free_ev};
        for (cudaEvent_t *ev : evs)
            if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess)
                return cuda_err(e, "event creation");
        for (int c = 0; c < CHUNKS; ++c)
            if ((e = cudaEventCreateWithFlags(&h.ev_a[c], cudaEventDisableTiming)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&h.ev_c[c], cudaEventDisableTiming)) != cudaSuccess)
                return cuda_err(e, "event creation");
        h.ready = true;
    }

    // device layout of one buffer set: A [M][K], SA [M][K/32], B [N][K], SB [N][K/32], C [M][ldcd]
    const int64_t kb = K / 32;
    const int64_t ldcd = (N + 7) / 8 * 8;                  // 16-byte rows for the vector stores
    const size_t off_sa = round256(static_cast<size_t>(M * K));
    const size_t off_b = off_sa + round256(static_cast<size_t>(M * kb));
    const size_t off_sb = off_b + round256(static_cast<size_t>(N * K));
    const size_t off_c = off_sb + round256(static_cast<size_t>(N * kb));
    const size_t need = off_c + round256(static_cast<size_t>(M * ldcd * 2));
    HostSet &bs = h.set[h.calls & 1];
    if (bs.bytes < need) {
        // the set may still be read by a download in flight: wait for it before freeing
        if (bs.used && (e = cudaEventSynchronize(bs.free_ev)) != cudaSuccess)
            return cuda_err(e, "waiting for a buffer set");
        if (bs.base) cudaFree(bs.base);
        bs.base = nullptr;
        bs.bytes = 0;
        if ((e = cudaMalloc(&bs.base, need)) != cudaSuccess) return cuda_err(e, "cudaMalloc");
        bs.bytes = need;
        bs.used = false;
    }
    uint8_t *dA = bs.base, *dSA = bs.base + off_sa, *dB = bs.base + off_b, *dSB = bs.base + off_sb;
    __half *dC = reinterpret_cast<__half *>(bs.base + off_c);
    cudaStream_t s = ctx.stream;

    // uploads: after the previous user of this set has been read back, and after the work already
    // on the caller's stream (the host planes may have been produced there)
    if ((e = cudaEventRecord(h.ev_start, s)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(h.up, h.ev_start, 0)) != cudaSuccess)
        return cuda_err(e, "ordering the uploads");
    if (bs.used && (e = cudaStreamWaitEvent(h.up, bs.free_ev, 0)) != cudaSuccess)
        return cuda_err(e, "ordering the uploads");
    auto up2d = [&](void *dst, int64_t dpitch, const void *src, int64_t spitch, int64_t width,
                    int64_t rows) {
        return cudaMemcpy2DAsync(dst, static_cast<size_t>(dpitch), src, static_cast<size_t>(spitch),
                                 static_cast<size_t>(width), static_cast<size_t>(rows),
                                 cudaMemcpyHostToDevice, h.up);
    };
    if (K > 0) {
        if ((e = up2d(dB, K, B->data, B->ld, K, N)) != cudaSuccess ||
            (e = up2d(dSB, kb, B->scales, B->lds, kb, N)) != cudaSuccess)
            return cuda_err(e, "upload of B");
    }
    if ((e = cudaEventRecord(h.ev_b, h.up)) != cudaSuccess) return cuda_err(e, "event record");
    // row chunks of A (multiples of 256 rows, the pair tile height)
    const int64_t step = ((M + CHUNKS - 1) / CHUNKS + 255) / 256 * 256;
    int nch = 0;
    for (int64_t r0 = 0; r0 < M; r0 += step, ++nch) {
        const int64_t rows = M - r0 < step ? M - r0 : step;
        if (K > 0) {
            if ((e = up2d(dA + r0 * K, K, A->data + r0 * A->ld, A->ld, K, rows)) != cudaSuccess ||
                (e = up2d(dSA + r0 * kb, kb, A->scales + r0 * A->lds, A->lds, kb, rows)) !=
                    cudaSuccess)
                return cuda_err(e, "upload of A");
        }
        if ((e = cudaEventRecord(h.ev_a[nch], h.up)) != cudaSuccess) return cuda_err(e, "event record");
    }

    // the product of each row chunk on the caller's stream, then its download.  On the CTA-pair
    // route B's scale plane is repacked once, right after B lands, and each chunk repacks only
    // its rows of A (into one buffer reused chunk after chunk: the stream orders them).
    if ((e = cudaStreamWaitEvent(s, h.ev_b, 0)) != cudaSuccess) return cuda_err(e, "ordering");
    const qgemm_tensor bc{QGEMM_E4M3, N, K, dB, K, dSB, kb};
    const qgemm_tensor a_first{QGEMM_E4M3, M < step ? M : step, K, dA, K, dSA, kb};
    const bool pair_b = K > 0 && N > 128;
    void *pack = nullptr;
    size_t pack_b_bytes = 0;
    if (pair_b) {
        pack_b_bytes = (qgi::mxfp8_pack_bytes(&bc) + 255) & ~size_t(255);
        if ((e = qgi::scratch_alloc(pack_b_bytes + qgi::mxfp8_pack_bytes(&a_first), ctx, &pack)) !=
            cudaSuccess)
            return cuda_err(e, "scale scratch");
        if ((e = qgi::launch_mxfp8_sf_pack(&bc, pack, ctx)) != cudaSuccess)
            return cuda_err(e, "scale repack of B");
    }
    nch = 0;
    for (int64_t r0 = 0; r0 < M; r0 += step, ++nch) {
        const int64_t rows = M - r0 < step ? M - r0 : step;
        if ((e = cudaStreamWaitEvent(s, h.ev_a[nch], 0)) != cudaSuccess) return cuda_err(e, "ordering");
        if (K == 0) {
            e = qgi::launch_fill_zero_f16(dC + r0 * ldcd, ldcd, rows, N, ctx);
        } else {
            const qgemm_tensor ac{QGEMM_E4M3, rows, K, dA + r0 * K, K, dSA + r0 * kb, kb};
            bool enc = true;
            if (pair_b && qgi::mxfp8_pair_eligible(&ac, &bc)) {
                uint8_t *pack_a = static_cast<uint8_t *>(pack) + pack_b_bytes;
                e = qgi::launch_mxfp8_sf_pack(&ac, pack_a, ctx);
                if (e == cudaSuccess)
                    e = qgi::launch_mxfp8_pair_packed(&ac, &bc, dC + r0 * ldcd, ldcd, pack_a, pack,
                                                      ctx, &enc);
            } else {
                // a K split only where the device call on the whole of A would split (A is one
                // chunk), so both calls sum in the same order and give the same bits
                e = qgi::launch_mxfp8(&ac, &bc, dC + r0 * ldcd, ldcd, ctx, &enc, rows == M);
            }
            if (!enc) return QGEMM_ERR_CUDA;
        }
        if (e != cudaSuccess) return cuda_err(e, "GEMM launch");
        if ((e = cudaEventRecord(h.ev_c[nch], s)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(h.down, h.ev_c[nch], 0)) != cudaSuccess)
            return cuda_err(e, "ordering the downloads");
        if ((e = cudaMemcpy2DAsync(static_cast<__half *>(C) + r0 * ldc,
                                   static_cast<size_t>(ldc) * 2, dC + r0 * ldcd,
                                   static_cast<size_t>(ldcd) * 2, static_cast<size_t>(N) * 2,
                                   static_cast<size_t>(rows), cudaMemcpyDeviceToHost,
                                   h.down)) != cudaSuccess)
            return cuda_err(e, "download of C");
    }
    if (pack && (e = qgi::scratch_free(pack, ctx)) != cudaSuccess)
        return cuda_err(e, "scale scratch");
    // the set is free once its downloads are done; the caller's stream completes with them
    if ((e = cudaEventRecord(bs.free_ev, h.down)) != cudaSuccess ||
        (e = cudaEventRecord(h.ev_out, h.down)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(s, h.ev_out, 0)) != cudaSuccess)
        return cuda_err(e, "ordering the end of the call");
    bs.used = true;
    ++h.calls;
    return QGEMM_OK;
}
