// dequant_debug.cu -- small utility kernels: the dequantise-only debug kernel, a zero fill for
// empty reductions, and the bounded-wait self test.
//
// The debug kernel writes out[r, k] = decode(data[r, k]) * 2^(scale[r, k/32] - 127) in fp32 so a
// test can compare the decoded operands bit for bit with the CPU reference (the check the
// "Running inline ML operations in a shader with Metal 4" sample makes against a CPU
// implementation).  E4M3 and E2M1 are decoded by the hardware conversion instructions (so the
// test also checks that the tensor cores' reading of the codes is the one the oracle spells out);
// integers by shifts.
#include <cuda_fp16.h>

#include "qgemm_internal.h"
#include "qgemm_ptx.cuh"

namespace {

using namespace qg;

__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
    uint32_t h2;
    const uint16_t pair = static_cast<uint16_t>(byte & 0xFF);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFF)));
}

// E2M1 nibble `hi` (0 = low, 1 = high) of `byte`.
__device__ __forceinline__ float e2m1_to_f32(uint32_t byte, int hi) {
    uint32_t h2;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t}"
        : "=r"(h2)
        : "r"(byte & 0xFFu));
    const uint16_t h = static_cast<uint16_t>(hi ? (h2 >> 16) : (h2 & 0xFFFF));
    return __half2float(__ushort_as_half(h));
}

__global__ void dequant_kernel(int dtype, int64_t rows, int64_t k, const uint8_t *__restrict__ data,
                               int64_t ld, const uint8_t *__restrict__ scales, int64_t lds,
                               float *__restrict__ out) {
    const int64_t total = rows * k;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / k, j = i - r * k;
        const uint8_t *row = data + r * ld;
        float v;
        if (dtype == QGEMM_F16) {
            v = __half2float(reinterpret_cast<const __half *>(row)[j]);
        } else {
            float q;
            if (dtype == QGEMM_E4M3) {
                q = e4m3_to_f32(row[j]);
            } else if (dtype == QGEMM_E2M1) {   // nibble (j & 1) of byte j / 2
                q = e2m1_to_f32(row[j >> 1], static_cast<int>(j & 1));
            } else if (dtype == QGEMM_INT8) {
                q = static_cast<float>(static_cast<int>(static_cast<int8_t>(row[j])));
            } else {  // int4: nibble (j & 1) of byte j / 2, sign-extended
                const uint32_t byte = row[j >> 1];
                const int nib = static_cast<int>((byte >> ((j & 1) * 4)) & 0xF);
                q = static_cast<float>(nib >= 8 ? nib - 16 : nib);
            }
            v = q * ue8m0_to_f32(scales[r * lds + (j >> 5)]);
        }
        out[i] = v;
    }
}

__global__ void fill_zero_f16_kernel(__half *C, int64_t ldc, int64_t M, int64_t N) {
    const int64_t total = M * N;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / N, c = i - r * N;
        C[r * ldc + c] = __ushort_as_half(0);
    }
}

// Epilogue of an empty reduction (K = 0) in accumulate mode: C = relu(C_old) in place.
__global__ void relu_inplace_f16_kernel(__half *C, int64_t ldc, int64_t M, int64_t N) {
    const int64_t total = M * N;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / N, c = i - r * N;
        __half *p = C + r * ldc + c;
        *p = __float2half_rn(fmaxf(__half2float(*p), 0.0f));
    }
}

// Waits on an mbarrier that nothing ever completes; the bounded wait must give up, record
// ERR_SELFTEST and let the kernel return normally.
__global__ void selftest_wait_kernel(unsigned *err, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(b, 0, timeout_ns)) atomicOr(err, ERR_SELFTEST);
    __syncthreads();
}

// One thread reads the SM cycle counter and the global nanosecond timer, naps in 0.5 us steps
// until window_ns of global time have passed (the timer always advances, so the loop ends), reads
// both again and stores out[0] = cycles, out[1] = nanoseconds.  The ratio is the SM clock over
// the window, whatever else the GPU runs meanwhile.  Launched as a programmatic dependent of the
// kernel before it on the stream, it runs beside that kernel when the kernel releases its
// dependents early (the library's GEMMs do) and then waits for it to complete, so that the
// probe's completion implies that kernel's.
__global__ void clock_probe_kernel(uint64_t window_ns, unsigned long long *out) {
    if (threadIdx.x == 0) {
        const uint64_t t0 = globaltimer_ns();
        const long long c0 = clock64();
        uint64_t t = t0;
        while (t - t0 < window_ns) {
            __nanosleep(500);
            t = globaltimer_ns();
        }
        const long long c1 = clock64();
        const uint64_t t1 = globaltimer_ns();
        out[0] = static_cast<unsigned long long>(c1 - c0);
        out[1] = static_cast<unsigned long long>(t1 - t0);
    }
    griddep_wait();
}

int grid_for(int64_t total, int num_sms) {
    int64_t g = (total + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (g > cap) g = cap;
    return g < 1 ? 1 : static_cast<int>(g);
}

}  // namespace

namespace qgi {

cudaError_t launch_dequant(const qgemm_tensor *t, float *out, const LaunchCtx &ctx) {
    const int64_t total = t->rows * t->k;
    if (total == 0) return cudaSuccess;
    dequant_kernel<<<grid_for(total, ctx.num_sms), 256, 0, ctx.stream>>>(
        t->dtype, t->rows, t->k, t->data, t->ld, t->scales, t->lds, out);
    return cudaGetLastError();
}

cudaError_t launch_fill_zero_f16(__half *C, int64_t ldc, int64_t M, int64_t N,
                                 const LaunchCtx &ctx) {
    if (M * N == 0) return cudaSuccess;
    fill_zero_f16_kernel<<<grid_for(M * N, ctx.num_sms), 256, 0, ctx.stream>>>(C, ldc, M, N);
    return cudaGetLastError();
}

cudaError_t launch_empty_sum_epilogue(__half *C, int64_t ldc, int64_t M, int64_t N,
                                      const LaunchCtx &ctx) {
    if (!(ctx.epi & EPI_ACCUMULATE)) return launch_fill_zero_f16(C, ldc, M, N, ctx);   // relu(0) = 0
    if (!(ctx.epi & EPI_RELU) || M * N == 0) return cudaSuccess;                        // C unchanged
    relu_inplace_f16_kernel<<<grid_for(M * N, ctx.num_sms), 256, 0, ctx.stream>>>(C, ldc, M, N);
    return cudaGetLastError();
}

cudaError_t launch_clock_probe(uint64_t window_ns, uint64_t *out, const LaunchCtx &ctx) {
    // A programmatic dependent: it starts only once every CTA of the kernel before it is running
    // (a probe launched on its own stream could take an SM first and hold back a CTA of a
    // persistent GEMM with a fixed tile order, which then waits for it).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = ctx.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, clock_probe_kernel, window_ns,
                              reinterpret_cast<unsigned long long *>(out));
}

cudaError_t launch_selftest_wait(uint64_t timeout_ns, const LaunchCtx &ctx) {
    selftest_wait_kernel<<<1, 32, 0, ctx.stream>>>(ctx.err, timeout_ns);
    return cudaGetLastError();
}

}  // namespace qgi
