// attention.cu -- fused attention forward, O = softmax(scale * Q K^T) V, fp16 in and out.
//
// "TensorOps: quantized matmul ...", section "FlashAttention on TensorOps (the recipe)", and
// "Optimize custom machine learning operations with Metal tensors", section on FlashAttention
// with cooperative tensors: one kernel computes Q K^T, takes each row's maximum, exponentiates
// the scores minus it and multiplies by V, and the intermediate matrix never goes to memory; the
// recipe gives each SIMD group whole rows so the row reduction needs no exchange, and feeds the
// exponentiated tile to the second product straight from registers when its layout allows.
//
// The GB300 form of that recipe:
//   * one CTA per (head, 128 query rows), head dimension 128; K and V tiles of 128 keys arrive
//     by TMA (3-D maps: d, row, head) into three stages of shared memory each, from two
//     producer threads (K runs ahead of V); a K stage is released when its scores are done, a
//     V stage when its P V is done;
//   * S = Q K^T for a key tile is one tcgen05.mma chain (M = 128 queries, N = 128 keys,
//     K = 128) into one of three 128-column TMEM buffers: the scores of tile j + 3 are issued
//     right after P V of tile j, so the softmax never waits for a P V -> S chain to drain;
//   * a TMEM lane is a query row, so each softmax thread owns a whole row: it reads its 128
//     scores into registers (tcgen05.ld), and the row maximum, the exponentials and the row sum
//     are in-register loops -- no exchange at all;
//   * the thread writes its row of P = exp2(s * scale * log2 e - m) as fp16 back into the same
//     TMEM columns (tcgen05.st) and the second product O += P V takes P as its A operand
//     straight from TMEM (the GB300 counterpart of passing the cooperative tensor as the left
//     input); V is read from shared memory as an MN-major operand (keys along K, d along N);
//   * the running maximum m is raised only when a tile's maximum exceeds it by more than 8 (in
//     log2 units); P then stays below 2^8 in fp16 and the rescale of O in TMEM (read, multiply,
//     write back, after the previous P V has completed) is rare;
//   * after the last tile each thread divides its row of O by its row sum and stores it.
// Keys past Lk (TMA zero fill) are masked to -inf; query rows past Lq are computed and dropped.
// Roles: warp 0 TMA producer of Q and K, warp 1 MMA issuer (one thread), warps 2-5 softmax and
// epilogue, warp 6 TMA producer of V.
// Every wait is bounded; on a timeout the kernel records the error bit, stops issuing work,
// waits for its MMAs, frees TMEM and returns.
#include "qgemm_common.cuh"
#include "qgemm_internal.h"
#include "qgemm_ptx.cuh"

namespace {

using namespace qg;

constexpr int BQ = 128;                 // query rows per CTA
constexpr int BKV = 128;                // keys per tile
constexpr int HD = 128;                 // head dimension
constexpr int KV_STAGES = 3;
constexpr int THREADS = 32 * 7;
constexpr uint32_t TMEM_COLS = 512;
constexpr int NSB = 3;                  // score buffers of 128 columns from column 0
constexpr uint32_t S_COL0 = 0;
constexpr uint32_t O_COL = 128 * NSB;   // output accumulator, 128 columns

constexpr uint32_t HALF_BYTES = 128 * 128;            // 128 rows x 64 halves (one swizzle span)
constexpr uint32_t TILE_BYTES = 2 * HALF_BYTES;       // 128 rows x 128 halves
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + TILE_BYTES;
constexpr uint32_t OFF_V = OFF_K + KV_STAGES * TILE_BYTES;
constexpr uint32_t OFF_BAR = OFF_V + KV_STAGES * TILE_BYTES;
// q_full, k_full[S], v_full[S], k_empty[S], v_empty[S], s_full[NSB], p_full[NSB],
// pv_done[NSB], drain, then the TMEM slot
constexpr int NBARS = 1 + 4 * KV_STAGES + 3 * NSB + 1;
constexpr uint32_t OFF_SLOT = OFF_BAR + NBARS * 8;
constexpr uint32_t SMEM_BYTES = OFF_SLOT + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// kind::f16, D fp32, A and B fp16, M = 128, N = 128.  S: both operands K-major.  P V: B (V) is
// MN-major (bit 16): keys run along K with a 128-byte row per key, d along N.
constexpr uint32_t IDESC_S = (1u << 4) | (static_cast<uint32_t>(128 >> 3) << 17) |
                             (static_cast<uint32_t>(128 >> 4) << 24);
constexpr uint32_t IDESC_PV = IDESC_S | (1u << 16);

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// One key tile of one query row: the running maximum m (log2 units) is given; writes
// P = 2^(s c - m) as fp16 pairs into TMEM columns scol .. scol + 63 of this warp's lanes and
// returns the row sum of P.  Every exponential is one ex2.approx (measured: moving a share of them
// to a cubic on the FMA pipe costs more issue slots than it saves).  MASK: keys >= valid give 0.
template <bool MASK>
__device__ __forceinline__ float softmax_tile(const uint32_t (&v)[128], int valid, float c,
                                              float m, uint32_t scol) {
    // row sum in four fp32 lanes (two packed pairs), scaled scores formed a pair at a time
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int h = 0; h < 2; ++h) {                      // 64 keys -> 32 packed columns
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int k0 = 64 * h + 2 * i;
            float x0, x1;
            fma2(x0, x1, __uint_as_float(v[k0]), __uint_as_float(v[k0 + 1]), c, c, -m, -m);
            float p0 = ex2_approx(x0);
            float p1 = ex2_approx(x1);
            if (MASK) {
                p0 = k0 < valid ? p0 : 0.0f;
                p1 = k0 + 1 < valid ? p1 : 0.0f;
            }
            const int a = 2 * (i & 1);
            add2(acc[a], acc[a + 1], p0, p1);
            pk[i] = pack_f16x2(p0, p1);
        }
        tmem_st_32x32b_x32(scol + 32 * h, pk);
    }
    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// Row maximum of the tile's raw scores; MASK: only keys < valid count.
template <bool MASK>
__device__ __forceinline__ float tile_max(const uint32_t (&v)[128], int valid) {
    float mx[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
    if constexpr (!MASK) {
        // three-input maximum: 64 instructions for the 128 scores, eight independent chains
#pragma unroll
        for (int i = 0; i < 128; i += 2) {
            const int k = (i >> 1) & 7;
            asm("max.f32 %0, %1, %2, %3;"
                : "=f"(mx[k])
                : "f"(mx[k]), "f"(__uint_as_float(v[i])), "f"(__uint_as_float(v[i + 1])));
        }
    } else {
#pragma unroll
        for (int i = 0; i < 128; ++i) {
            const float x = __uint_as_float(v[i]);
            mx[i & 7] = fmaxf(mx[i & 7], i < valid ? x : -INFINITY);
        }
    }
    return fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
}

__global__ void __launch_bounds__(THREADS, 1)
attention_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, __half *__restrict__ O, int64_t o_hs,
                 int64_t o_rs, int Lq, int Lk, float c_log2, unsigned *err, uint64_t timeout_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_1024(smem_raw);
    const uint32_t sb = smem_u32(smem);
    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    const int head = blockIdx.y;
    const int q0 = blockIdx.x * BQ;
    const int nkv = (Lk + BKV - 1) / BKV;

    const uint32_t q_full = sb + OFF_BAR;
    auto k_full = [&](int s) { return sb + OFF_BAR + 8u * (1 + s); };
    auto v_full = [&](int s) { return sb + OFF_BAR + 8u * (1 + KV_STAGES + s); };
    auto k_empty = [&](int s) { return sb + OFF_BAR + 8u * (1 + 2 * KV_STAGES + s); };
    auto v_empty = [&](int s) { return sb + OFF_BAR + 8u * (1 + 3 * KV_STAGES + s); };
    auto s_full = [&](int b) { return sb + OFF_BAR + 8u * (1 + 4 * KV_STAGES + b); };
    auto p_full = [&](int b) { return sb + OFF_BAR + 8u * (1 + 4 * KV_STAGES + NSB + b); };
    auto pv_done = [&](int b) { return sb + OFF_BAR + 8u * (1 + 4 * KV_STAGES + 2 * NSB + b); };
    const uint32_t drain_bar = sb + OFF_BAR + 8u * (1 + 4 * KV_STAGES + 3 * NSB);
    volatile uint32_t *slot = reinterpret_cast<volatile uint32_t *>(smem + OFF_SLOT);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < KV_STAGES; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(v_full(s), 1);
            mbar_init(k_empty(s), 1);
            mbar_init(v_empty(s), 1);
        }
        for (int b = 0; b < NSB; ++b) {
            mbar_init(s_full(b), 1);
            mbar_init(p_full(b), 4);     // one arrival per softmax warp
            mbar_init(pv_done(b), 1);
        }
        mbar_init(drain_bar, 1);
        fence_barrier_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(const_cast<uint32_t *>(slot)), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *slot;

    if (warp == 0) {
        // ------------------------------------------------------ producer of Q and K
        if (lane == 0) {
            bool ok = true;
            mbar_arrive_expect_tx(q_full, TILE_BYTES);
            tma_load_3d(sb + OFF_Q, &tmQ, q_full, 0, q0, head);
            tma_load_3d(sb + OFF_Q + HALF_BYTES, &tmQ, q_full, 64, q0, head);
            int issued = 0;
            for (int j = 0; j < nkv; ++j) {
                const int st = j % KV_STAGES;
                if (!mbar_wait(k_empty(st), ((j / KV_STAGES) & 1) ^ 1, timeout_ns)) {
                    ok = false;
                    break;
                }
                const uint32_t sk = sb + OFF_K + st * TILE_BYTES;
                mbar_arrive_expect_tx(k_full(st), TILE_BYTES);
                tma_load_3d(sk, &tmK, k_full(st), 0, j * BKV, head);
                tma_load_3d(sk + HALF_BYTES, &tmK, k_full(st), 64, j * BKV, head);
                ++issued;
            }
            if (!ok) atomicOr(err, ERR_PRODUCER);
            // no copy may be in flight when the CTA exits
            bool drained = mbar_wait(q_full, 0, timeout_ns);
            for (int i = max(0, issued - KV_STAGES); i < issued && drained; ++i)
                drained = mbar_wait(k_full(i % KV_STAGES), (i / KV_STAGES) & 1, timeout_ns);
            if (!drained) atomicOr(err, ERR_DRAIN);
        }
        __syncwarp();
    } else if (warp == 6) {
        // ----------------------------------------------------------- producer of V
        if (lane == 0) {
            bool ok = true;
            int issued = 0;
            for (int j = 0; j < nkv; ++j) {
                const int st = j % KV_STAGES;
                if (!mbar_wait(v_empty(st), ((j / KV_STAGES) & 1) ^ 1, timeout_ns)) {
                    ok = false;
                    break;
                }
                const uint32_t sv = sb + OFF_V + st * TILE_BYTES;
                mbar_arrive_expect_tx(v_full(st), TILE_BYTES);
                tma_load_3d(sv, &tmV, v_full(st), 0, j * BKV, head);
                tma_load_3d(sv + HALF_BYTES, &tmV, v_full(st), 64, j * BKV, head);
                ++issued;
            }
            if (!ok) atomicOr(err, ERR_PRODUCER);
            bool drained = true;
            for (int i = max(0, issued - KV_STAGES); i < issued && drained; ++i)
                drained = mbar_wait(v_full(i % KV_STAGES), (i / KV_STAGES) & 1, timeout_ns);
            if (!drained) atomicOr(err, ERR_DRAIN);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // --------------------------------------------------------- MMA issuer
            const uint64_t qdesc = smem_desc(sb + OFF_Q, 16, 1024, SWZ_128B);
            bool ok = mbar_wait(q_full, 0, timeout_ns);
            auto issue_s = [&](int j) -> bool {
                const int b = j % NSB, st = j % KV_STAGES;
                if (!mbar_wait(k_full(st), (j / KV_STAGES) & 1, timeout_ns)) return false;
                tc_fence_after();
                const uint64_t kdesc = smem_desc(sb + OFF_K + st * TILE_BYTES, 16, 1024, SWZ_128B);
#pragma unroll
                for (uint32_t kk = 0; kk < HD / 16; ++kk) {
                    // 16 of d per MMA: span kk / 4 (64 halves each), 32 bytes kk % 4 into it
                    const uint64_t off = (kk >> 2) * (HALF_BYTES >> 4) + 2 * (kk & 3);
                    mma_f16(tmem_base + S_COL0 + 128 * b, qdesc + off, kdesc + off, IDESC_S,
                            kk > 0 ? 1u : 0u);
                }
                tc_commit(s_full(b));
                tc_commit(k_empty(st));
                return true;
            };
            auto issue_pv = [&](int j) -> bool {
                const int b = j % NSB, st = j % KV_STAGES;
                if (!mbar_wait(p_full(b), (j / NSB) & 1, timeout_ns)) return false;
                if (!mbar_wait(v_full(st), (j / KV_STAGES) & 1, timeout_ns)) return false;
                tc_fence_after();
                const uint32_t sv = sb + OFF_V + st * TILE_BYTES;
#pragma unroll
                for (uint32_t kk = 0; kk < BKV / 16; ++kk) {
                    // keys 16 kk .. 16 kk + 15: P columns 8 kk.. (two fp16 per column); V rows
                    // start 16 kk x 128 bytes into each span; the second 64 of d is the other
                    // span (leading offset), the next 8 keys 1024 bytes on (stride offset)
                    const uint64_t vdesc = smem_desc(sv + kk * 2048, HALF_BYTES, 1024, SWZ_128B);
                    mma_f16_ta(tmem_base + O_COL, tmem_base + S_COL0 + 128 * b + 8 * kk, vdesc,
                               IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(v_empty(st));
                tc_commit(pv_done(b));
                return true;
            };
            // scores run NSB tiles ahead: S(0 .. NSB-1), then P V(j) followed by S(j + NSB),
            // which reuses the buffer P V(j) has just read (the tensor pipe keeps issue order)
            for (int j = 0; j < NSB && j < nkv && ok; ++j) ok = issue_s(j);
            for (int j = 0; j < nkv && ok; ++j) {
                if (!issue_pv(j)) {
                    ok = false;
                    break;
                }
                if (j + NSB < nkv && !issue_s(j + NSB)) ok = false;
            }
            if (!ok) atomicOr(err, ERR_MMA);
            tc_commit(drain_bar);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- softmax and epilogue
        const uint32_t q = warp & 3;                          // TMEM lane quarter
        const uint32_t lq = (q * 32) << 16;                   // lane field of this warp's rows
        const int row = q0 + static_cast<int>(q * 32 + lane);
        float m_used = -INFINITY, l = 0.0f;
        bool ok = true;
        for (int j = 0; j < nkv; ++j) {
            const int b = j % NSB;
            if (!mbar_wait(s_full(b), (j / NSB) & 1, timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t v[BKV];
            const uint32_t scol = tmem_base + lq + S_COL0 + 128 * b;
#pragma unroll
            for (int ch = 0; ch < BKV / 32; ++ch)
                tmem_ld_32x32b_x32(scol + 32 * ch, *reinterpret_cast<uint32_t(*)[32]>(&v[32 * ch]));
            tmem_wait_ld();
            const int valid = Lk - j * BKV;                   // keys of this tile inside Lk
            const bool full = valid >= BKV;
            const float mx2 = (full ? tile_max<false>(v, valid) : tile_max<true>(v, valid)) * c_log2;
            // raise the running maximum only when this tile exceeds it by more than 2^8
            const bool need = mx2 > m_used + 8.0f;
            if (__any_sync(0xFFFFFFFFu, need)) {
                const float m_new = fmaxf(m_used, mx2);
                if (j > 0) {
                    // the previous P V must have completed before O is rescaled
                    if (!mbar_wait(pv_done((j - 1) % NSB), ((j - 1) / NSB) & 1, timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const float alpha = ex2_approx(m_used - m_new);
                    const uint32_t ocol = tmem_base + lq + O_COL;
#pragma unroll 1
                    for (int ch = 0; ch < HD / 32; ++ch) {
                        uint32_t o[32];
                        tmem_ld_32x32b_x32(ocol + 32 * ch, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st_32x32b_x32(ocol + 32 * ch, o);
                    }
                    tmem_wait_st();
                    l *= alpha;
                }
                m_used = m_new;
            }
            l += full ? softmax_tile<false>(v, valid, c_log2, m_used, scol)
                      : softmax_tile<true>(v, valid, c_log2, m_used, scol);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(b));
        }
        if (!ok) {
            if (lane == 0) atomicOr(err, ERR_EPILOGUE);
        } else if (nkv > 0) {
            const int last = nkv - 1;
            if (!mbar_wait(pv_done(last % NSB), (last / NSB) & 1, timeout_ns)) {
                if (lane == 0) atomicOr(err, ERR_EPILOGUE);
            } else {
                tc_fence_after();
                const float inv = 1.0f / l;
                const uint32_t ocol = tmem_base + lq + O_COL;
                __half *orow = O + static_cast<int64_t>(head) * o_hs + static_cast<int64_t>(row) * o_rs;
#pragma unroll 1
                for (int ch = 0; ch < HD / 32; ++ch) {
                    uint32_t o[32];
                    tmem_ld_32x32b_x32(ocol + 32 * ch, o);
                    tmem_wait_ld();
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[i] = pack_f16x2(__uint_as_float(o[2 * i]) * inv,
                                           __uint_as_float(o[2 * i + 1]) * inv);
                    if (row < Lq) {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * ch);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        // every MMA that writes this CTA's TMEM has completed before it is freed
        if (!mbar_wait(drain_bar, 0, timeout_ns) && lane == 0) atomicOr(err, ERR_DRAIN);
        __syncwarp();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace

namespace qgi {

cudaError_t launch_attention(const AttnArgs &a, const LaunchCtx &ctx, bool *encode_ok) {
    CUtensorMap tmQ, tmK, tmV;
    *encode_ok =
        encode_tma_3d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.Q, HD, a.Lq, a.BH, a.q_rs * 2,
                      a.q_hs * 2, 64, BQ, 1, CU_TENSOR_MAP_SWIZZLE_128B) &&
        encode_tma_3d(&tmK, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.K, HD, a.Lk, a.BH, a.k_rs * 2,
                      a.k_hs * 2, 64, BKV, 1, CU_TENSOR_MAP_SWIZZLE_128B) &&
        encode_tma_3d(&tmV, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.V, HD, a.Lk, a.BH, a.v_rs * 2,
                      a.v_hs * 2, 64, BKV, 1, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!*encode_ok) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(attention_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const float c_log2 = a.scale * 1.4426950408889634f;
    const dim3 grid(static_cast<unsigned>((a.Lq + BQ - 1) / BQ), static_cast<unsigned>(a.BH));
    attention_kernel<<<grid, THREADS, SMEM_BYTES, ctx.stream>>>(tmQ, tmK, tmV, a.O, a.o_hs, a.o_rs,
                                                                a.Lq, a.Lk, c_log2, ctx.err,
                                                                ctx.timeout_ns);
    return cudaGetLastError();
}

}  // namespace qgi
