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
//   * one CTA per (head, 256 query rows), held as two query tiles of 128 rows, head dimension
//     128; K and V tiles of 128 keys arrive by TMA (3-D maps: d, row, head) from two producer
//     threads (three K stages, two V stages), each shared by both query tiles;
//   * TMEM holds, per query tile t, a 128-column score buffer S_t and a 128-column output
//     accumulator O_t.  S_t = Q_t K_j^T is one tcgen05.mma chain (M = N = K = 128);
//   * a TMEM lane is a query row, so each softmax thread owns a whole row: it takes the row's
//     maximum over the tile's 128 scores, writes P = exp2(s * scale * log2 e - m) as fp16 back
//     over its own scores (tcgen05.st), and the second product O_t += P V_j takes P as its A
//     operand straight from TMEM (the GB300 counterpart of passing the cooperative tensor as
//     the left input); V is read from shared memory as an MN-major operand;
//   * two softmax warpgroups, one per query tile, alternate with the tensor pipe: the MMA warp
//     issues, per key tile, P V for tile 0 and the next scores of tile 0, then the same for tile
//     1, so while one warpgroup exponentiates its scores the tensor pipe works for the other.
//     The softmax releases P in two halves of 64 keys; P V of the first half runs while it
//     exponentiates the second.  The whole MMA warp runs the loop and one
//     elected lane issues (measured on GB300: a lone thread issues a tcgen05.mma in about 57
//     cycles, an elected lane of a converged warp in about 14, and the pipe queues about 8 MMAs
//     of 128 x 128 x 16 ahead); the waits before a block test their barriers together, so
//     their latencies overlap;
//   * the running maximum m is raised only when a tile's maximum exceeds it by more than 8 (in
//     log2 units); P then stays below 2^8 in fp16 and the rescale of O_t in TMEM (read, multiply,
//     write back) is rare.  It needs no extra wait: the commit that reports S_t(j) ready also
//     covers every MMA issued before it, P V of tile j - 1 included.  The first half of P is
//     computed with m as it stands while the tile's maximum is taken; only when the maximum
//     moves is it computed again;
//   * after the last key tile each thread divides its row of O by its row sum and stores it.
// Keys past Lk (TMA zero fill) are masked to -inf; query rows past Lq are computed and dropped.
// Roles: warp 0 TMA producer of Q and K, warp 1 MMA issuer (one elected lane) and TMEM owner,
// warp 2 TMA producer of V, warp 3 idle, warps 4-7 softmax of query tile 0, warps 8-11 of query
// tile 1
// (warp w reads TMEM lane quarter w % 4).
// Every wait is bounded; on a timeout the kernel records the error bit, stops issuing work,
// waits for its MMAs, frees TMEM and returns.
#include "qgemm_common.cuh"
#include "qgemm_internal.h"
#include "qgemm_ptx.cuh"

namespace {

using namespace qg;

constexpr int BQ = 128;                 // query rows per query tile
constexpr int QT = 2;                   // query tiles per CTA
constexpr int BKV = 128;                // keys per tile
constexpr int HD = 128;                 // head dimension
constexpr int K_STAGES = 3;
constexpr int V_STAGES = 2;
constexpr int SOFTMAX_WARP0 = 4;
constexpr int THREADS = 32 * (SOFTMAX_WARP0 + 4 * QT);
constexpr uint32_t TMEM_COLS = 512;
__host__ __device__ constexpr uint32_t s_col(int t) { return 128u * t; }          // S_t
__host__ __device__ constexpr uint32_t o_col(int t) { return 128u * (QT + t); }   // O_t

constexpr uint32_t HALF_BYTES = 128 * 128;            // 128 rows x 64 halves (one swizzle span)
constexpr uint32_t TILE_BYTES = 2 * HALF_BYTES;       // 128 rows x 128 halves
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + QT * TILE_BYTES;
constexpr uint32_t OFF_V = OFF_K + K_STAGES * TILE_BYTES;
constexpr uint32_t OFF_BAR = OFF_V + V_STAGES * TILE_BYTES;
// q_full, k_full[K], k_empty[K], v_full[V], v_empty[V], s_full[QT], p_full[QT][2] (keys 0..63,
// 64..127), o_done[QT],
// drain, then the TMEM slot
constexpr int NBARS = 1 + 2 * K_STAGES + 2 * V_STAGES + 4 * QT + 1;
constexpr uint32_t OFF_SLOT = OFF_BAR + NBARS * 8;
constexpr uint32_t SMEM_BYTES = OFF_SLOT + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(QT == 2, "the MMA issue order is written for two query tiles");

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

// 64 keys of one query row (key k0 + i of the tile in v[i]): P = 2^(s c - m) as 32 fp16 pairs
// in pk; returns their sum.  Every exponential is one ex2.approx (measured: taking a share of
// them from a polynomial on the FMA pipe makes the softmax slower, not faster).  MASK: keys >=
// valid give 0.
template <bool MASK>
__device__ __forceinline__ float exp_half(const uint32_t (&v)[64], int k0, int valid, float c,
                                          float m, uint32_t (&pk)[32]) {
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        float x0, x1;
        fma2(x0, x1, __uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]), c, c, -m, -m);
        float p0 = ex2_approx(x0);
        float p1 = ex2_approx(x1);
        if (MASK) {
            p0 = k0 + 2 * i < valid ? p0 : 0.0f;
            p1 = k0 + 2 * i + 1 < valid ? p1 : 0.0f;
        }
        const int a = 2 * (i & 1);
        add2(acc[a], acc[a + 1], p0, p1);
        pk[i] = pack_f16x2(p0, p1);
    }
    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// Maximum of 64 raw scores (keys k0 .. k0 + 63 of the tile); MASK: only keys < valid count.
template <bool MASK>
__device__ __forceinline__ float half_max(const uint32_t (&v)[64], int k0, int valid) {
    float mx[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
    if constexpr (!MASK) {
        // three-input maximum: 32 instructions for the 64 scores, eight independent chains
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
            const int k = (i >> 1) & 7;
            asm("max.f32 %0, %1, %2, %3;"
                : "=f"(mx[k])
                : "f"(mx[k]), "f"(__uint_as_float(v[i])), "f"(__uint_as_float(v[i + 1])));
        }
    } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            const float x = __uint_as_float(v[i]);
            mx[i & 7] = fmaxf(mx[i & 7], k0 + i < valid ? x : -INFINITY);
        }
    }
    return fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
}

// Partial rows a half of a split unit leaves for attention_merge_kernel: the unnormalised O of
// its 256 rows (fp32, row-major), then their running maxima m (log2 units), then their sums l.
constexpr int UNIT_ROWS = QT * BQ;
constexpr size_t WS_FLOATS_PER_HALF = static_cast<size_t>(UNIT_ROWS) * (HD + 2);

__global__ void __launch_bounds__(THREADS, 1)
attention_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, __half *__restrict__ O, int64_t o_hs,
                 int64_t o_rs, int Lq, int Lk, float c_log2, int nqb, int n_direct, int kv_split,
                 float *__restrict__ ws, unsigned *err, uint64_t timeout_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_1024(smem_raw);
    const uint32_t sb = smem_u32(smem);
    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    // A unit is (head, 256 query rows).  CTAs below n_direct take one unit over all its key
    // tiles; the rest come in pairs that split one unit's key tiles at kv_split (the last wave of
    // a grid that would leave SMs idle) and leave their partial rows in ws.
    const int nkv_all = (Lk + BKV - 1) / BKV;
    const int s_idx = static_cast<int>(blockIdx.x) - n_direct;   // >= 0: a half of a split unit
    const int unit = s_idx < 0 ? static_cast<int>(blockIdx.x) : n_direct + (s_idx >> 1);
    const int kv_half = s_idx < 0 ? -1 : (s_idx & 1);
    const int head = unit / nqb;
    const int q0 = (unit - head * nqb) * UNIT_ROWS;
    const int kv0 = kv_half == 1 ? kv_split : 0;                 // first key tile of this CTA
    const int nkv = kv_half < 0 ? nkv_all : (kv_half == 0 ? kv_split : nkv_all - kv_split);

    const uint32_t q_full = sb + OFF_BAR;
    auto k_full = [&](int s) { return sb + OFF_BAR + 8u * (1 + s); };
    auto k_empty = [&](int s) { return sb + OFF_BAR + 8u * (1 + K_STAGES + s); };
    auto v_full = [&](int s) { return sb + OFF_BAR + 8u * (1 + 2 * K_STAGES + s); };
    auto v_empty = [&](int s) { return sb + OFF_BAR + 8u * (1 + 2 * K_STAGES + V_STAGES + s); };
    constexpr int B0 = 1 + 2 * K_STAGES + 2 * V_STAGES;
    auto s_full = [&](int t) { return sb + OFF_BAR + 8u * (B0 + t); };
    auto p_full = [&](int t, int h) { return sb + OFF_BAR + 8u * (B0 + QT + 2 * t + h); };
    auto o_done = [&](int t) { return sb + OFF_BAR + 8u * (B0 + 3 * QT + t); };
    const uint32_t drain_bar = sb + OFF_BAR + 8u * (B0 + 4 * QT);
    volatile uint32_t *slot = reinterpret_cast<volatile uint32_t *>(smem + OFF_SLOT);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < K_STAGES; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(k_empty(s), 1);
        }
        for (int s = 0; s < V_STAGES; ++s) {
            mbar_init(v_full(s), 1);
            mbar_init(v_empty(s), 1);
        }
        for (int t = 0; t < QT; ++t) {
            mbar_init(s_full(t), 1);
            mbar_init(p_full(t, 0), 4);   // one arrival per softmax warp of the tile
            mbar_init(p_full(t, 1), 4);
            mbar_init(o_done(t), 1);
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

    // warpgroup 0 (producers, MMA issuer) needs few registers; the softmax warpgroups hold a row
    // of 128 scores each: 72 x 128 + 208 x 256 <= 168 x 384, the registers the block is launched
    // with.  One reallocation per warpgroup, outside the role branches.
    if (warp < SOFTMAX_WARP0) {
        regs_release<72>();
        if (warp == 0) {
            // ------------------------------------------------------ producer of Q and K
            if (lane == 0) {
                bool ok = true;
                mbar_arrive_expect_tx(q_full, QT * TILE_BYTES);
                for (int t = 0; t < QT; ++t) {
                    tma_load_3d(sb + OFF_Q + t * TILE_BYTES, &tmQ, q_full, 0, q0 + t * BQ, head);
                    tma_load_3d(sb + OFF_Q + t * TILE_BYTES + HALF_BYTES, &tmQ, q_full, 64, q0 + t * BQ,
                                head);
                }
                int issued = 0;
                for (int j = 0; j < nkv; ++j) {
                    const int st = j % K_STAGES;
                    if (!mbar_wait(k_empty(st), ((j / K_STAGES) & 1) ^ 1, timeout_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sk = sb + OFF_K + st * TILE_BYTES;
                    mbar_arrive_expect_tx(k_full(st), TILE_BYTES);
                    tma_load_3d(sk, &tmK, k_full(st), 0, (kv0 + j) * BKV, head);
                    tma_load_3d(sk + HALF_BYTES, &tmK, k_full(st), 64, (kv0 + j) * BKV, head);
                    ++issued;
                }
                if (!ok) atomicOr(err, ERR_PRODUCER);
                // no copy may be in flight when the CTA exits
                bool drained = mbar_wait(q_full, 0, timeout_ns);
                for (int i = max(0, issued - K_STAGES); i < issued && drained; ++i)
                    drained = mbar_wait(k_full(i % K_STAGES), (i / K_STAGES) & 1, timeout_ns);
                if (!drained) atomicOr(err, ERR_DRAIN);
            }
            __syncwarp();
        } else if (warp == 2) {
            // ----------------------------------------------------------- producer of V
            if (lane == 0) {
                bool ok = true;
                int issued = 0;
                for (int j = 0; j < nkv; ++j) {
                    const int st = j % V_STAGES;
                    if (!mbar_wait(v_empty(st), ((j / V_STAGES) & 1) ^ 1, timeout_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sv = sb + OFF_V + st * TILE_BYTES;
                    mbar_arrive_expect_tx(v_full(st), TILE_BYTES);
                    tma_load_3d(sv, &tmV, v_full(st), 0, (kv0 + j) * BKV, head);
                    tma_load_3d(sv + HALF_BYTES, &tmV, v_full(st), 64, (kv0 + j) * BKV, head);
                    ++issued;
                }
                if (!ok) atomicOr(err, ERR_PRODUCER);
                bool drained = true;
                for (int i = max(0, issued - V_STAGES); i < issued && drained; ++i)
                    drained = mbar_wait(v_full(i % V_STAGES), (i / V_STAGES) & 1, timeout_ns);
                if (!drained) atomicOr(err, ERR_DRAIN);
            }
            __syncwarp();
        } else if (warp == 1) {
            // ----------------------------------------------------------------- MMA issuer
            // The whole warp runs the loop and waits; one elected lane issues (a loop run by one
            // lane alone issues measurably slower).
            bool ok = mbar_wait_warp(q_full, 0, timeout_ns);
            const uint64_t qdesc0 = smem_desc(sb + OFF_Q, 16, 1024, SWZ_128B);
            const uint64_t kdesc0 = smem_desc(sb + OFF_K, 16, 1024, SWZ_128B);
            // V's descriptor: keys 16 kk .. 16 kk + 15 start 16 kk x 128 bytes into each span,
            // the second 64 of d is the other span (leading offset), the next 8 keys 1024 bytes
            // on (stride offset).
            const uint64_t vdesc0 = smem_desc(sb + OFF_V, HALF_BYTES, 1024, SWZ_128B);
            // The descriptors and TMEM addresses are formed by the whole warp, outside the
            // issuing branch: formed inside it, measured, each MMA issues much more slowly.
            const uint64_t qdesc[QT] = {qdesc0, qdesc0 + (TILE_BYTES >> 4)};
            const uint32_t scol_t[QT] = {tmem_base + s_col(0), tmem_base + s_col(1)};
            const uint32_t ocol_t[QT] = {tmem_base + o_col(0), tmem_base + o_col(1)};
            auto mma_s = [&](int t, uint64_t kdesc) {   // S_t = Q_t K^T
#pragma unroll
                for (uint32_t kk = 0; kk < HD / 16; ++kk) {
                    // 16 of d per MMA: span kk / 4 (64 halves each), 32 bytes kk % 4 into it
                    const uint64_t off = (kk >> 2) * (HALF_BYTES >> 4) + 2 * (kk & 3);
                    mma_f16(scol_t[t], qdesc[t] + off, kdesc + off, IDESC_S, kk > 0 ? 1u : 0u);
                }
            };
            // O_t (+)= P_t V over keys 64 h .. 64 h + 63, P_t in S_t's columns 32 h ..
            auto mma_pv = [&](int t, int h, uint64_t vdesc, bool acc) {
#pragma unroll
                for (uint32_t k4 = 0; k4 < BKV / 32; ++k4) {   // keys 16 kk ..: P columns 8 kk ..
                    const uint32_t kk = 4 * h + k4;
                    mma_f16_ta(ocol_t[t], scol_t[t] + 8 * kk, vdesc + kk * (2048 >> 4), IDESC_PV,
                               (acc || kk > 0) ? 1u : 0u);
                }
            };
            // S_0(0), S_1(0); then per key tile j two blocks, each behind its waits: P V of query
            // tile 0 with its scores for key tile j + 1, then the same for query tile 1.  The
            // tensor pipe's queue is short: a thread issuing into a full queue stalls until it
            // drains, and every wait, fence and commit that follows leaves the pipe idle, so the
            // blocks are as few and as long as the dependencies allow.  The scores S_t(j + 1)
            // overwrite the P that P V has just read: the tensor pipe executes one thread's MMAs
            // in issue order.
            if (nkv > 0) {
                ok = ok && mbar_wait_warp(k_full(0), 0, timeout_ns);
                if (ok && elect_one()) {
                    mma_s(0, kdesc0);
                    tc_commit(s_full(0));
                    mma_s(1, kdesc0);
                    tc_commit(s_full(1));
                    tc_commit(k_empty(0));
                }
                __syncwarp();
            }
            for (int j = 0; j < nkv && ok; ++j) {
                const bool next = j + 1 < nkv;
                const int kn = (j + 1) % K_STAGES;
                // the three barriers are tested at once (their latencies overlap); only when one
                // is not ready does the warp wait on each in turn
                const uint32_t vb = v_full(j % V_STAGES), vp = (j / V_STAGES) & 1;
                const uint32_t kb = k_full(kn), kp = ((j + 1) / K_STAGES) & 1;
                const bool r_v = mbar_try_wait(vb, vp);
                const bool r_p = mbar_try_wait(p_full(0, 0), j & 1);
                const bool r_k = !next || mbar_try_wait(kb, kp);
                if (!__all_sync(0xFFFFFFFFu, r_v && r_p && r_k))
                    ok = mbar_wait_warp(vb, vp, timeout_ns) &&
                         mbar_wait_warp(p_full(0, 0), j & 1, timeout_ns) &&
                         (!next || mbar_wait_warp(kb, kp, timeout_ns));
                if (!ok) break;
                tc_fence_after();
                const int vs = j % V_STAGES;
                const uint64_t vdesc = vdesc0 + static_cast<uint64_t>(vs) * (TILE_BYTES >> 4);
                const uint64_t kdesc = kdesc0 + static_cast<uint64_t>(kn) * (TILE_BYTES >> 4);
                // the first half of P V while the softmax exponentiates the second half
                if (elect_one()) mma_pv(0, 0, vdesc, j > 0);
                __syncwarp();
                ok = mbar_wait_warp(p_full(0, 1), j & 1, timeout_ns);
                if (!ok) break;
                tc_fence_after();
                if (elect_one()) {
                    mma_pv(0, 1, vdesc, true);
                    if (next) {
                        mma_s(0, kdesc);
                        tc_commit(s_full(0));
                    } else {
                        tc_commit(o_done(0));
                    }
                }
                __syncwarp();
                ok = mbar_wait_warp(p_full(1, 0), j & 1, timeout_ns);
                if (!ok) break;
                tc_fence_after();
                if (elect_one()) mma_pv(1, 0, vdesc, j > 0);
                __syncwarp();
                ok = mbar_wait_warp(p_full(1, 1), j & 1, timeout_ns);
                if (!ok) break;
                tc_fence_after();
                if (elect_one()) {
                    mma_pv(1, 1, vdesc, true);
                    tc_commit(v_empty(vs));
                    if (next) {
                        mma_s(1, kdesc);
                        tc_commit(s_full(1));
                        tc_commit(k_empty(kn));
                    } else {
                        tc_commit(o_done(1));
                    }
                }
                __syncwarp();
            }
            if (elect_one()) {
                if (!ok) atomicOr(err, ERR_MMA);
                tc_commit(drain_bar);
            }
            __syncwarp();
        }
    } else {
        regs_claim<208>();
        // ------------------------------------------------------- softmax and epilogue
        const int t = static_cast<int>(warp - SOFTMAX_WARP0) >> 2;   // query tile
        const uint32_t q = warp & 3;                                  // TMEM lane quarter
        const uint32_t lq = (q * 32) << 16;                           // lane field of these rows
        const int row = q0 + t * BQ + static_cast<int>(q * 32 + lane);
        const uint32_t scol = tmem_base + lq + s_col(t);
        const uint32_t ocol = tmem_base + lq + o_col(t);
        float m_used = -INFINITY, l = 0.0f;
        bool ok = true;
        for (int j = 0; j < nkv; ++j) {
            if (!mbar_wait(s_full(t), j & 1, timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int valid = Lk - (kv0 + j) * BKV;           // keys of this tile inside Lk
            const bool full = valid >= BKV;
            // the whole row of scores in registers: one TMEM round trip per tile
            uint32_t v[128];
            tmem_ld_32x32b_x32(scol, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            tmem_ld_32x32b_x32(scol + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            tmem_ld_32x32b_x32(scol + 64, *reinterpret_cast<uint32_t(*)[32]>(&v[64]));
            tmem_ld_32x32b_x32(scol + 96, *reinterpret_cast<uint32_t(*)[32]>(&v[96]));
            tmem_wait_ld();
            const uint32_t(&v0)[64] = *reinterpret_cast<const uint32_t(*)[64]>(&v[0]);
            const uint32_t(&v1)[64] = *reinterpret_cast<const uint32_t(*)[64]>(&v[64]);
            // P of keys 0 .. 63 under the running maximum as it stands, computed while the tile's
            // maximum is taken (the exponentials are bound by the MUFU pipe, the maximum fills
            // issue slots beside them): the maximum is off the path to the first P V
            uint32_t pk[32];
            float l0 = full ? exp_half<false>(v0, 0, valid, c_log2, m_used, pk)
                            : exp_half<true>(v0, 0, valid, c_log2, m_used, pk);
            const float mx = full ? fmaxf(half_max<false>(v0, 0, valid), half_max<false>(v1, 64, valid))
                                  : fmaxf(half_max<true>(v0, 0, valid), half_max<true>(v1, 64, valid));
            const float mx2 = mx * c_log2;
            // the running maximum is raised only when this tile exceeds it by more than 8 (log2
            // units; always on the first tile): then O_t and l are rescaled and P recomputed
            const bool need = mx2 > m_used + 8.0f;
            if (__any_sync(0xFFFFFFFFu, need)) {
                const float m_new = fmaxf(m_used, mx2);
                if (j > 0) {
                    // P V of key tile j - 1 has completed: the commit behind s_full covers it
                    const float alpha = ex2_approx(m_used - m_new);
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
                l0 = full ? exp_half<false>(v0, 0, valid, c_log2, m_used, pk)
                          : exp_half<true>(v0, 0, valid, c_log2, m_used, pk);
            }
            // P over the scores: keys 0 .. 63 into columns 0 .. 31, released to P V at once, then
            // keys 64 .. 127 into columns 32 .. 63
            l += l0;
            tmem_st_32x32b_x32(scol, pk);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(t, 0));
            l += full ? exp_half<false>(v1, 64, valid, c_log2, m_used, pk)
                      : exp_half<true>(v1, 64, valid, c_log2, m_used, pk);
            tmem_st_32x32b_x32(scol + 32, pk);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(t, 1));
        }
        if (!ok) {
            if (lane == 0) atomicOr(err, ERR_EPILOGUE);
        } else if (nkv > 0) {
            if (!mbar_wait(o_done(t), 0, timeout_ns)) {
                if (lane == 0) atomicOr(err, ERR_EPILOGUE);
            } else if (kv_half >= 0) {
                // a half of a split unit: the row's unnormalised O, m and l for the merge
                tc_fence_after();
                float *wsb = ws + static_cast<size_t>(s_idx) * WS_FLOATS_PER_HALF;
                const int r = t * BQ + static_cast<int>(q * 32 + lane);
                float4 *dst = reinterpret_cast<float4 *>(wsb + static_cast<size_t>(r) * HD);
#pragma unroll 1
                for (int ch = 0; ch < HD / 32; ++ch) {
                    uint32_t o[32];
                    tmem_ld_32x32b_x32(ocol + 32 * ch, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[8 * ch + i] = make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]),
                                                      __uint_as_float(o[4 * i + 2]), __uint_as_float(o[4 * i + 3]));
                }
                wsb[static_cast<size_t>(UNIT_ROWS) * HD + r] = m_used;
                wsb[static_cast<size_t>(UNIT_ROWS) * (HD + 1) + r] = l;
            } else {
                tc_fence_after();
                const float inv = 1.0f / l;
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

// Rows of the split units: O = (a0 O0 + a1 O1) / (a0 l0 + a1 l1) with a_h = 2^(m_h - max(m0, m1)),
// the two halves' partial rows combined as the running-maximum recurrence combines key tiles.
// One warp per row, four columns per lane.
__global__ void __launch_bounds__(256)
attention_merge_kernel(const float *__restrict__ ws, int n_direct, int n_split, int nqb,
                       __half *__restrict__ O, int64_t o_hs, int64_t o_rs, int Lq) {
    const int slot = static_cast<int>(blockIdx.x) * 8 + static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31);
    const int su = slot / UNIT_ROWS, r = slot - su * UNIT_ROWS;
    if (su >= n_split) return;
    const int unit = n_direct + su;
    const int head = unit / nqb;
    const int row = (unit - head * nqb) * UNIT_ROWS + r;
    if (row >= Lq) return;
    const float *w0 = ws + static_cast<size_t>(2 * su) * WS_FLOATS_PER_HALF;
    const float *w1 = w0 + WS_FLOATS_PER_HALF;
    const size_t im = static_cast<size_t>(UNIT_ROWS) * HD + r;
    const size_t il = static_cast<size_t>(UNIT_ROWS) * (HD + 1) + r;
    const float m = fmaxf(w0[im], w1[im]);
    const float a0 = exp2f(w0[im] - m), a1 = exp2f(w1[im] - m);
    const float inv = 1.0f / (a0 * w0[il] + a1 * w1[il]);
    const float4 o0 = reinterpret_cast<const float4 *>(w0 + static_cast<size_t>(r) * HD)[lane];
    const float4 o1 = reinterpret_cast<const float4 *>(w1 + static_cast<size_t>(r) * HD)[lane];
    const uint32_t p0 = pack_f16x2((a0 * o0.x + a1 * o1.x) * inv, (a0 * o0.y + a1 * o1.y) * inv);
    const uint32_t p1 = pack_f16x2((a0 * o0.z + a1 * o1.z) * inv, (a0 * o0.w + a1 * o1.w) * inv);
    __half *dst = O + static_cast<int64_t>(head) * o_hs + static_cast<int64_t>(row) * o_rs + 4 * lane;
    *reinterpret_cast<uint2 *>(dst) = make_uint2(p0, p1);
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
    // Units (head, 256 query rows) fill whole waves of one CTA per SM; when the last wave would
    // leave at least half the SMs idle, its units are split in two along the keys, a CTA each,
    // and merged afterwards: that wave then takes half the time.
    const int nqb = (a.Lq + UNIT_ROWS - 1) / UNIT_ROWS;
    const int64_t units = static_cast<int64_t>(nqb) * a.BH;
    const int nkv_all = (a.Lk + BKV - 1) / BKV;
    const int64_t rem = ctx.num_sms > 0 ? units % ctx.num_sms : 0;
    const int n_split =
        (units > ctx.num_sms && rem > 0 && 2 * rem <= ctx.num_sms && nkv_all >= 4)
            ? static_cast<int>(rem) : 0;
    const int64_t n_direct = units - n_split;
    if (n_direct + 2 * n_split > 0x7FFFFFFF) return cudaErrorInvalidValue;
    float *ws = nullptr;
    if (n_split > 0) {
        e = scratch_alloc(2 * n_split * WS_FLOATS_PER_HALF * sizeof(float), ctx,
                          reinterpret_cast<void **>(&ws));
        if (e != cudaSuccess) return e;
    }
    const unsigned grid = static_cast<unsigned>(n_direct + 2 * n_split);
    attention_kernel<<<grid, THREADS, SMEM_BYTES, ctx.stream>>>(
        tmQ, tmK, tmV, a.O, a.o_hs, a.o_rs, a.Lq, a.Lk, c_log2, nqb, static_cast<int>(n_direct),
        nkv_all / 2, ws, ctx.err, ctx.timeout_ns);
    e = cudaGetLastError();
    if (n_split > 0) {
        if (e == cudaSuccess) {
            const unsigned mgrid = static_cast<unsigned>((n_split * UNIT_ROWS + 7) / 8);
            attention_merge_kernel<<<mgrid, 256, 0, ctx.stream>>>(
                ws, static_cast<int>(n_direct), n_split, nqb, a.O, a.o_hs, a.o_rs, a.Lq);
            e = cudaGetLastError();
        }
        const cudaError_t f = scratch_free(ws, ctx);
        if (e == cudaSuccess) e = f;
    }
    return e;
}

}  // namespace qgi
