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
//   * the work is the sequence of units (head, 256 query rows), each over its key tiles of 128
//     keys, on one CTA per SM (persistent).  Whole waves run data-parallel (unit w G + c on CTA
//     c in wave w) while at least two waves' worth remain, so the CTAs at work at one time read
//     the K and V of few heads and L2 keeps them; the key tiles of the units left (one to two
//     waves' worth) are shared out in equal, contiguous ranges, one per CTA (they differ by at
//     most one key tile), so no wave is left part-empty.  A CTA's share of one unit is a part:
//     whole, the unit's tail (the range starts inside the unit) or its head (the range ends
//     inside it).  A tail part leaves its unnormalised rows, running maxima and sums in a
//     workspace and raises a flag; the CTA holding the unit's head merges them into its own
//     rows when it writes the output, the way the running-maximum recurrence combines key
//     tiles.  A tail is the first part of its CTA's range and a head the last, so a head's
//     partners have long finished when it gets there; the CTAs wait on one another only there,
//     and the launch is cooperative (every CTA resident);
//   * a unit is held as two query tiles of 128 rows, head dimension 128; K and V tiles arrive
//     by TMA (3-D maps: d, row, head) from two producer threads (three K stages, two V stages),
//     each shared by both query tiles, and run on across part boundaries; a third producer
//     loads each part's Q, a query tile as soon as the last part's output has left its buffer;
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
//   * after a part's last key tile each thread divides its row of O by its row sum (merged with
//     the tail parts' for a head part) and writes it, as fp16, into the query tile's Q buffer in
//     the output tensor map's layout; one lane per warp stores its 32 rows with bulk tensor
//     copies.  A tail part writes its rows in fp32, lane-interleaved so each store is one
//     contiguous 512-byte run.
// Keys past Lk (TMA zero fill) are masked to -inf; query rows past Lq are computed and dropped.
// Roles: warp 0 TMA producer of K, warp 1 MMA issuer (one elected lane) and TMEM owner, warp 2
// TMA producer of V, warp 3 TMA producer of Q, warps 4-7 softmax of query tile 0, warps 8-11 of
// query tile 1 (warp w reads TMEM lane quarter w % 4).
// Every wait is bounded; on a timeout the kernel records the error bit, stops issuing work,
// waits for its copies and MMAs, frees TMEM and returns.
#include "qgemm_common.cuh"
#include "qgemm_debug.cuh"
#include "qgemm_internal.h"
#include "qgemm_ptx.cuh"

namespace {

using namespace qg;

constexpr int BQ = 128;                 // query rows per query tile
constexpr int QT = 2;                   // query tiles per unit
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
// q_full[QT], q_free[QT], k_full[K], k_empty[K], v_full[V], v_empty[V], s_full[QT],
// p_full[QT][2] (keys 0..63, 64..127), o_done[QT], drain, then the TMEM slot
constexpr int NBARS = 2 * QT + 2 * K_STAGES + 2 * V_STAGES + 4 * QT + 1;
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

// 3-D tiled bulk tensor store shared -> global (bulk-group completion); the parts of the box
// outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const void *tmap, uint32_t src, int32_t c0, int32_t c1,
                                             int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(tmap)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// L2 prefetch of one 3-D TMA box (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_3d(const void *tmap, int32_t c0, int32_t c1,
                                                int32_t c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

__device__ __forceinline__ void st_release_gpu(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Waits (bounded) until another CTA has raised the flag; false on a timeout.
__device__ __forceinline__ bool wait_flag(const unsigned *f, uint64_t timeout_ns) {
    if (ld_acquire_gpu(f) != 0) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        __nanosleep(128);
        if (ld_acquire_gpu(f) != 0) return true;
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
}

constexpr int UNIT_ROWS = QT * BQ;
// A tail part's rows in the workspace (one slot per CTA, fp32): O of its 256 rows as eight
// 32-row slabs (slab k = 4 t + lane quarter, the rows of one softmax warp), each slab as
// [column group of 4][row of the slab][4 columns], so a warp's store of one column group is 512
// contiguous bytes; then the rows' running maxima m (log2 units), then their sums l.
constexpr size_t WS_F4_PER_SLAB = (HD / 4) * 32;
constexpr size_t WS_M = static_cast<size_t>(UNIT_ROWS) * HD;
constexpr size_t WS_L = WS_M + UNIT_ROWS;
constexpr size_t WS_FLOATS = WS_L + UNIT_ROWS;
constexpr int FLAGS_PER_SLOT = UNIT_ROWS / 32;   // one per slab (per writing warp)

// First key tile of CTA c's range when T tiles are shared by G CTAs (the first T % G ranges
// take one tile more).
__host__ __device__ __forceinline__ int64_t range_start(int64_t c, int64_t T, int64_t G) {
    const int64_t b = T / G, r = T % G;
    return c * b + (c < r ? c : r);
}

// Whole waves of units run data-parallel (wave w: unit w G + c on CTA c) while at least two
// waves remain, so the CTAs at work at one time read the K and V of few heads and L2 keeps
// them; the key tiles of the units left (one to two waves' worth) are shared out in ranges.
__host__ __device__ __forceinline__ int64_t dp_waves(int64_t units, int64_t G) {
    return units / G >= 2 ? units / G - 1 : 0;
}

enum PartKind { PART_WHOLE = 0, PART_TAIL = 1, PART_HEAD = 2 };
struct Part {
    int64_t unit;
    int head, q0, kv0, nkv, kind;
};
// One CTA's work: its data-parallel units, then its range [begin, end) of the T key tiles of
// the units from u0 on.
struct Sched {
    int64_t G, cta, D, u0, T, begin, end;
    int nkv_all, nqb;
};
__device__ __forceinline__ Sched make_sched(int64_t units, int nkv_all, int nqb) {
    Sched s;
    s.G = gridDim.x;
    s.cta = blockIdx.x;
    s.D = dp_waves(units, s.G);
    s.u0 = s.D * s.G;
    s.T = (units - s.u0) * nkv_all;
    s.begin = range_start(s.cta, s.T, s.G);
    s.end = range_start(s.cta + 1, s.T, s.G);
    s.nkv_all = nkv_all;
    s.nqb = nqb;
    return s;
}
// Position in the CTA's work: data-parallel units done, then the key-tile cursor of the range.
struct Cursor {
    int64_t dp, cur;
};
__device__ __forceinline__ Cursor cursor_start(const Sched &s) { return Cursor{0, s.begin}; }
// The next part, or false when the CTA's work is done.
__device__ __forceinline__ bool next_part(const Sched &s, Cursor &c, Part &p) {
    if (c.dp < s.D) {
        p.unit = c.dp * s.G + s.cta;
        p.kv0 = 0;
        p.nkv = s.nkv_all;
        p.kind = PART_WHOLE;
        ++c.dp;
    } else if (c.cur < s.end) {
        const int64_t u = c.cur / s.nkv_all;
        p.unit = s.u0 + u;
        p.kv0 = static_cast<int>(c.cur - u * s.nkv_all);
        const int64_t uend = (u + 1) * s.nkv_all;
        p.nkv = static_cast<int>((s.end < uend ? s.end : uend) - c.cur);
        p.kind = p.kv0 > 0 ? PART_TAIL : (s.end < uend ? PART_HEAD : PART_WHOLE);
        c.cur += p.nkv;
    } else {
        return false;
    }
    p.head = static_cast<int>(p.unit / s.nqb);
    p.q0 = static_cast<int>(p.unit - static_cast<int64_t>(p.head) * s.nqb) * UNIT_ROWS;
    return true;
}

__global__ void __launch_bounds__(THREADS, 1)
attention_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                 int Lq, int Lk, float c_log2, int nqb, int64_t units, float *ws,
                 unsigned *flags, unsigned *err, uint64_t timeout_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_1024(smem_raw);
    const uint32_t sb = smem_u32(smem);
    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    // Every role walks the CTA's parts in the same order.  The K and V rings and the score / P
    // barriers run on across part boundaries (their phases follow a key-tile count over the
    // whole range), so the next part's K and V loads overlap the last part's end; its Q waits
    // for the last part's output to leave the Q buffer.
    const int nkv_all = (Lk + BKV - 1) / BKV;
    const Sched sc = make_sched(units, nkv_all, nqb);

    auto q_full = [&](int t) { return sb + OFF_BAR + 8u * t; };
    auto q_free = [&](int t) { return sb + OFF_BAR + 8u * (QT + t); };
    constexpr int B1 = 2 * QT;
    auto k_full = [&](int s) { return sb + OFF_BAR + 8u * (B1 + s); };
    auto k_empty = [&](int s) { return sb + OFF_BAR + 8u * (B1 + K_STAGES + s); };
    auto v_full = [&](int s) { return sb + OFF_BAR + 8u * (B1 + 2 * K_STAGES + s); };
    auto v_empty = [&](int s) { return sb + OFF_BAR + 8u * (B1 + 2 * K_STAGES + V_STAGES + s); };
    constexpr int B0 = B1 + 2 * K_STAGES + 2 * V_STAGES;
    auto s_full = [&](int t) { return sb + OFF_BAR + 8u * (B0 + t); };
    auto p_full = [&](int t, int h) { return sb + OFF_BAR + 8u * (B0 + QT + 2 * t + h); };
    auto o_done = [&](int t) { return sb + OFF_BAR + 8u * (B0 + 3 * QT + t); };
    const uint32_t drain_bar = sb + OFF_BAR + 8u * (B0 + 4 * QT);
    static_assert(B0 + 4 * QT + 1 == NBARS, "barrier count");
    volatile uint32_t *slot = reinterpret_cast<volatile uint32_t *>(smem + OFF_SLOT);

    if (threadIdx.x == 0) {
        for (int t = 0; t < QT; ++t) {
            mbar_init(q_full(t), 1);
            mbar_init(q_free(t), 4);   // one arrival per softmax warp of the tile
        }
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
            mbar_init(p_full(t, 0), 4);
            mbar_init(p_full(t, 1), 4);
            mbar_init(o_done(t), 1);
        }
        mbar_init(drain_bar, 1);
        fence_barrier_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmO);
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
    // of 128 scores each: 88 x 128 + 208 x 256 <= 168 x 384, the registers the block is launched
    // with.  One reallocation per warpgroup, outside the role branches.
    if (warp < SOFTMAX_WARP0) {
        regs_release<88>();
        if (warp == 3) {
            // ------------------------------------------------------------ producer of Q
            // Query tile t of a part is loaded once the last part's output has left the tile's
            // buffer (q_free: its softmax warps stage the output there); the next part's Q is
            // prefetched into L2 meanwhile.
            if (lane == 0) {
                bool ok = true;
                uint32_t armed[QT] = {0, 0};   // parts loaded per query tile
                Cursor cs = cursor_start(sc);
                Part p;
                while (ok && next_part(sc, cs, p)) {
                    for (int t = 0; t < QT; ++t) {
                        if (armed[t] > 0 && !mbar_wait(q_free(t), (armed[t] - 1) & 1, timeout_ns)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(q_full(t), TILE_BYTES);
                        const uint32_t dst = sb + OFF_Q + t * TILE_BYTES;
                        tma_load_3d(dst, &tmQ, q_full(t), 0, p.q0 + t * BQ, p.head);
                        tma_load_3d(dst + HALF_BYTES, &tmQ, q_full(t), 64, p.q0 + t * BQ, p.head);
                        ++armed[t];
                    }
                    Cursor nc = cs;
                    Part nx;
                    if (ok && next_part(sc, nc, nx)) {
                        for (int t = 0; t < QT; ++t) {
                            tma_prefetch_3d(&tmQ, 0, nx.q0 + t * BQ, nx.head);
                            tma_prefetch_3d(&tmQ, 64, nx.q0 + t * BQ, nx.head);
                        }
                    }
                }
                if (!ok) atomicOr(err, ERR_PRODUCER);
                // no copy may be in flight when the CTA exits
                bool drained = true;
                for (int t = 0; t < QT && drained; ++t)
                    if (armed[t] > 0)
                        drained = mbar_wait(q_full(t), (armed[t] - 1) & 1, timeout_ns);
                if (!drained) atomicOr(err, ERR_DRAIN);
            }
            __syncwarp();
        } else if (warp == 0 || warp == 2) {
            // ------------------------------------------------ producers of K (warp 0), V (2)
            if (lane == 0) {
                const bool isk = warp == 0;
                const int stages = isk ? K_STAGES : V_STAGES;
                const CUtensorMap *tm = isk ? &tmK : &tmV;
                const uint32_t off = isk ? OFF_K : OFF_V;
                bool ok = true;
                // stage and phase advance per key tile over the whole range
                int st = 0;
                uint32_t ph = 0, armed = 0, last_ph = 0;   // armed: bit per stage
                Cursor cs = cursor_start(sc);
                Part p;
                while (ok && next_part(sc, cs, p)) {
                    for (int j = 0; j < p.nkv; ++j) {
                        const uint32_t full = isk ? k_full(st) : v_full(st);
                        const uint32_t empty = isk ? k_empty(st) : v_empty(st);
                        // debug build: the key tile starts inside Lk
                        if (!QG_IN_BOUNDS(err, (p.kv0 + j) * BKV < Lk) ||
                            !mbar_wait(empty, ph ^ 1, timeout_ns)) {
                            ok = false;
                            break;
                        }
                        const uint32_t dst = sb + off + st * TILE_BYTES;
                        mbar_arrive_expect_tx(full, TILE_BYTES);
                        tma_load_3d(dst, tm, full, 0, (p.kv0 + j) * BKV, p.head);
                        tma_load_3d(dst + HALF_BYTES, tm, full, 64, (p.kv0 + j) * BKV, p.head);
                        armed |= 1u << st;
                        last_ph = (last_ph & ~(1u << st)) | (ph << st);
                        if (++st == stages) {
                            st = 0;
                            ph ^= 1;
                        }
                    }
                }
                if (!ok) atomicOr(err, ERR_PRODUCER);
                // no copy may be in flight when the CTA exits
                bool drained = true;
                for (int x = 0; x < stages && drained; ++x)
                    if (armed >> x & 1)
                        drained = mbar_wait(isk ? k_full(x) : v_full(x), last_ph >> x & 1,
                                            timeout_ns);
                if (!drained) atomicOr(err, ERR_DRAIN);
            }
            __syncwarp();
        } else if (warp == 1) {
            // ----------------------------------------------------------------- MMA issuer
            // The whole warp runs the loop and waits; one elected lane issues (a loop run by one
            // lane alone issues measurably slower).  Per key tile: P V of query tile 0 (its first
            // half as soon as the softmax releases keys 0 .. 63) with tile 0's next scores, then
            // the same for tile 1.  The scores S_t(j + 1) overwrite the P that P V has just read:
            // the tensor pipe executes one thread's MMAs in issue order.  A part's first P V
            // (accumulate off) overwrites O_t only after the softmax warps, which read the last
            // part's O_t first, have released that part's first P.
            const uint64_t qdesc0 = smem_desc(sb + OFF_Q, 16, 1024, SWZ_128B);
            const uint64_t kdesc0 = smem_desc(sb + OFF_K, 16, 1024, SWZ_128B);
            // V's descriptor: keys 16 kk .. 16 kk + 15 start 16 kk x 128 bytes into each span,
            // the second 64 of d is the other span (leading offset), the next 8 keys 1024 bytes
            // on (stride offset).
            const uint64_t vdesc0 = smem_desc(sb + OFF_V, HALF_BYTES, 1024, SWZ_128B);
            // descriptors and TMEM addresses are formed by the whole warp, outside the issuing
            // branch: formed inside it, measured, each MMA issues much more slowly
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
            bool ok = true;
            // ring positions advance per key tile over the whole range: the K tile to consume
            // next, the V tile of the current key tile; gp: the key tile's score / P phase; qp:
            // the part's Q phase
            int ks = 0, vs = 0;
            uint32_t kph = 0, vph = 0, gp = 0, qp = 0;
            Cursor cs = cursor_start(sc);
            Part p;
            for (; ok && next_part(sc, cs, p); qp ^= 1) {
                // S_0(0) once Q_0 and the part's first K tile are in, then S_1(0)
                ok = mbar_wait_warp(q_full(0), qp, timeout_ns) &&
                     mbar_wait_warp(k_full(ks), kph, timeout_ns);
                if (!ok) break;
                tc_fence_after();
                uint64_t kdesc = kdesc0 + static_cast<uint64_t>(ks) * (TILE_BYTES >> 4);
                if (elect_one()) {
                    mma_s(0, kdesc);
                    tc_commit(s_full(0));
                }
                __syncwarp();
                ok = mbar_wait_warp(q_full(1), qp, timeout_ns);
                if (!ok) break;
                tc_fence_after();
                if (elect_one()) {
                    mma_s(1, kdesc);
                    tc_commit(s_full(1));
                    tc_commit(k_empty(ks));
                }
                __syncwarp();
                if (++ks == K_STAGES) {
                    ks = 0;
                    kph ^= 1;
                }
                for (int j = 0; j < p.nkv && ok; ++j, gp ^= 1) {
                    const bool next = j + 1 < p.nkv;
                    // the three barriers are tested at once (their latencies overlap); only when
                    // one is not ready does the warp wait on each in turn
                    const uint32_t vb = v_full(vs), kb = k_full(ks);
                    const bool r_v = mbar_try_wait(vb, vph);
                    const bool r_p = mbar_try_wait(p_full(0, 0), gp);
                    const bool r_k = !next || mbar_try_wait(kb, kph);
                    if (!__all_sync(0xFFFFFFFFu, r_v && r_p && r_k))
                        ok = mbar_wait_warp(vb, vph, timeout_ns) &&
                             mbar_wait_warp(p_full(0, 0), gp, timeout_ns) &&
                             (!next || mbar_wait_warp(kb, kph, timeout_ns));
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t vdesc = vdesc0 + static_cast<uint64_t>(vs) * (TILE_BYTES >> 4);
                    kdesc = kdesc0 + static_cast<uint64_t>(ks) * (TILE_BYTES >> 4);
                    // the first half of P V while the softmax exponentiates the second half
                    if (elect_one()) mma_pv(0, 0, vdesc, j > 0);
                    __syncwarp();
                    ok = mbar_wait_warp(p_full(0, 1), gp, timeout_ns);
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
                    ok = mbar_wait_warp(p_full(1, 0), gp, timeout_ns);
                    if (!ok) break;
                    tc_fence_after();
                    if (elect_one()) mma_pv(1, 0, vdesc, j > 0);
                    __syncwarp();
                    ok = mbar_wait_warp(p_full(1, 1), gp, timeout_ns);
                    if (!ok) break;
                    tc_fence_after();
                    if (elect_one()) {
                        mma_pv(1, 1, vdesc, true);
                        tc_commit(v_empty(vs));
                        if (next) {
                            mma_s(1, kdesc);
                            tc_commit(s_full(1));
                            tc_commit(k_empty(ks));
                        } else {
                            tc_commit(o_done(1));
                        }
                    }
                    __syncwarp();
                    if (++vs == V_STAGES) {
                        vs = 0;
                        vph ^= 1;
                    }
                    if (next && ++ks == K_STAGES) {
                        ks = 0;
                        kph ^= 1;
                    }
                }
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
        const int slab = t * 4 + static_cast<int>(q);                // 32-row slab of the unit
        const int r = slab * 32 + static_cast<int>(lane);            // row within the unit
        const uint32_t scol = tmem_base + lq + s_col(t);
        const uint32_t ocol = tmem_base + lq + o_col(t);
        // this warp's 32 output rows, staged in the query tile's buffer
        const uint32_t stage = sb + OFF_Q + t * TILE_BYTES + q * 32 * 128;
        bool ok = true;
        uint32_t gp = 0, qp = 0;   // key-tile and part phases
        Cursor cs = cursor_start(sc);
        Part p;
        for (; ok && next_part(sc, cs, p); qp ^= 1) {
            float m_used = -INFINITY, l = 0.0f;
            for (int j = 0; j < p.nkv; ++j, gp ^= 1) {
                if (!mbar_wait(s_full(t), gp, timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int valid = Lk - (p.kv0 + j) * BKV;   // keys of this tile inside Lk
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
                // P of keys 0 .. 63 under the running maximum as it stands, computed while the
                // tile's maximum is taken (the exponentials are bound by the MUFU pipe, the
                // maximum fills issue slots beside them): the maximum is off the path to the
                // first P V
                uint32_t pk[32];
                float l0 = full ? exp_half<false>(v0, 0, valid, c_log2, m_used, pk)
                                : exp_half<true>(v0, 0, valid, c_log2, m_used, pk);
                const float mx =
                    full ? fmaxf(half_max<false>(v0, 0, valid), half_max<false>(v1, 64, valid))
                         : fmaxf(half_max<true>(v0, 0, valid), half_max<true>(v1, 64, valid));
                const float mx2 = mx * c_log2;
                // the running maximum is raised only when this tile exceeds it by more than 8
                // (log2 units; always on the part's first tile): then O_t and l are rescaled and
                // P recomputed
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
                            for (int x = 0; x < 32; ++x)
                                o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
                            tmem_st_32x32b_x32(ocol + 32 * ch, o);
                        }
                        tmem_wait_st();
                        l *= alpha;
                    }
                    m_used = m_new;
                    l0 = full ? exp_half<false>(v0, 0, valid, c_log2, m_used, pk)
                              : exp_half<true>(v0, 0, valid, c_log2, m_used, pk);
                }
                // P over the scores: keys 0 .. 63 into columns 0 .. 31, released to P V at once,
                // then keys 64 .. 127 into columns 32 .. 63
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
            if (!ok) break;
            // The part's O_t is complete, and so is every MMA that read Q (o_done covers them);
            // the issuer meanwhile runs on into the next part, whose first P V (overwriting O_t)
            // waits for this warp's first P arrival, after the reads below.
            if (!mbar_wait(o_done(t), qp, timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // debug build: a part that shares its unit with another CTA has the workspace and
            // flags the host allocates when some range starts inside a unit
            if (p.kind != PART_WHOLE && !QG_IN_BOUNDS(err, ws != nullptr && flags != nullptr)) {
                ok = false;
                break;
            }
            if (p.kind == PART_TAIL) {
                // the unit's tail: unnormalised rows, m and l for the CTA holding its head
                float *wsb = ws + static_cast<size_t>(sc.cta) * WS_FLOATS;
                float4 *dst = reinterpret_cast<float4 *>(wsb) + slab * WS_F4_PER_SLAB + lane;
#pragma unroll 1
                for (int ch = 0; ch < HD / 32; ++ch) {
                    uint32_t o[32];
                    tmem_ld_32x32b_x32(ocol + 32 * ch, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int x = 0; x < 8; ++x)
                        dst[(8 * ch + x) * 32] =
                            make_float4(__uint_as_float(o[4 * x]), __uint_as_float(o[4 * x + 1]),
                                        __uint_as_float(o[4 * x + 2]), __uint_as_float(o[4 * x + 3]));
                }
                wsb[WS_M + r] = m_used;
                wsb[WS_L + r] = l;
                // the rows are visible before the flag
                __threadfence();
                __syncwarp();
                if (lane == 0) st_release_gpu(flags + sc.cta * FLAGS_PER_SLOT + slab, 1u);
            } else {
                // Whole unit, or its head merged with the tails the next CTAs computed: with
                // m = max(m_own, m_w ...), O = (a_own O_own + sum a_w O_w) / (a_own l + sum a_w l_w),
                // a = 2^(m_part - m).
                const int64_t w0 = sc.cta + 1;
                int64_t w_end = w0;   // tail parts: CTAs w0 .. w_end - 1
                float m_tot = m_used;
                if (p.kind == PART_HEAD) {
                    const int64_t uend = (p.unit - sc.u0 + 1) * nkv_all;
                    while (w_end < sc.G && range_start(w_end, sc.T, sc.G) < uend) ++w_end;
                    for (int64_t w = w0; w < w_end && ok; ++w) {
                        // debug build: the writer's range starts inside this unit
                        ok = QG_IN_BOUNDS(err, range_start(w, sc.T, sc.G) >
                                                   (p.unit - sc.u0) * nkv_all) &&
                             wait_flag(flags + w * FLAGS_PER_SLOT + slab, timeout_ns);
                        if (ok) m_tot = fmaxf(m_tot, __ldcg(ws + w * WS_FLOATS + WS_M + r));
                    }
                    if (!__all_sync(0xFFFFFFFFu, ok)) {
                        ok = false;
                        break;
                    }
                }
                const float a_own = exp2f(m_used - m_tot);
                float lsum = a_own * l;
                for (int64_t w = w0; w < w_end; ++w) {
                    const float *wsb = ws + w * WS_FLOATS;
                    lsum += exp2f(__ldcg(wsb + WS_M + r) - m_tot) * __ldcg(wsb + WS_L + r);
                }
                const float inv = 1.0f / lsum;
                // The normalised rows go out through shared memory, in the layout of the output
                // tensor map (two spans of 64 columns, 128 bytes a row, 16-byte chunks swizzled
                // by the row), and one lane stores them with two bulk tensor copies.  Each lane
                // writing its own row straight to global memory touched 32 lines per store and
                // was measured to take several times as long.
#pragma unroll 1
                for (int ch = 0; ch < HD / 32; ++ch) {
                    uint32_t o[32];
                    tmem_ld_32x32b_x32(ocol + 32 * ch, o);
                    tmem_wait_ld();
                    float f[32];
#pragma unroll
                    for (int x = 0; x < 32; ++x) f[x] = __uint_as_float(o[x]) * a_own;
                    for (int64_t w = w0; w < w_end; ++w) {
                        const float *wsb = ws + w * WS_FLOATS;
                        const float a_w = exp2f(__ldcg(wsb + WS_M + r) - m_tot);
                        const float4 *src =
                            reinterpret_cast<const float4 *>(wsb) + slab * WS_F4_PER_SLAB + lane;
#pragma unroll
                        for (int x = 0; x < 8; ++x) {
                            const float4 y = __ldcg(src + (8 * ch + x) * 32);
                            f[4 * x] += a_w * y.x;
                            f[4 * x + 1] += a_w * y.y;
                            f[4 * x + 2] += a_w * y.z;
                            f[4 * x + 3] += a_w * y.w;
                        }
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) pk[x] = pack_f16x2(f[2 * x] * inv, f[2 * x + 1] * inv);
                    // columns 32 ch .. 32 ch + 31: span ch / 2, chunks 4 (ch % 2) .. + 3 of the row
                    const uint32_t rowb = stage + (ch >> 1) * HALF_BYTES + lane * 128;
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const uint32_t c = 4 * (ch & 1) + x;
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                         rowb + ((c ^ (lane & 7)) << 4)),
                                     "r"(pk[4 * x]), "r"(pk[4 * x + 1]), "r"(pk[4 * x + 2]),
                                     "r"(pk[4 * x + 3])
                                     : "memory");
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                const int row0 = p.q0 + t * BQ + static_cast<int>(q * 32);
                if (lane == 0 && row0 < Lq) {
                    tma_store_3d(&tmO, stage, 0, row0, p.head);
                    tma_store_3d(&tmO, stage + HALF_BYTES, 64, row0, p.head);
                    bulk_commit();
                    // the copies have read the buffer before Q may be loaded into it again
                    bulk_wait_read<0>();
                }
                __syncwarp();
            }
            // the query tile's buffer is free for the next part's Q
            if (lane == 0) mbar_arrive(q_free(t));
        }
        if (!ok && lane == 0) atomicOr(err, ERR_EPILOGUE);
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
    CUtensorMap tmQ, tmK, tmV, tmO;
    *encode_ok =
        encode_tma_3d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.Q, HD, a.Lq, a.BH, a.q_rs * 2,
                      a.q_hs * 2, 64, BQ, 1, CU_TENSOR_MAP_SWIZZLE_128B) &&
        encode_tma_3d(&tmK, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.K, HD, a.Lk, a.BH, a.k_rs * 2,
                      a.k_hs * 2, 64, BKV, 1, CU_TENSOR_MAP_SWIZZLE_128B) &&
        encode_tma_3d(&tmV, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.V, HD, a.Lk, a.BH, a.v_rs * 2,
                      a.v_hs * 2, 64, BKV, 1, CU_TENSOR_MAP_SWIZZLE_128B) &&
        encode_tma_3d(&tmO, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.O, HD, a.Lq, a.BH, a.o_rs * 2,
                      a.o_hs * 2, 64, 32, 1, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!*encode_ok) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(attention_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const float c_log2 = a.scale * 1.4426950408889634f;
    // The key tiles of all units, shared out in equal ranges over one CTA per SM; a range of
    // fewer than MIN_RANGE tiles is not worth a part's fixed cost, so small problems take fewer
    // CTAs.
    constexpr int64_t MIN_RANGE = 4;
    const int nqb = (a.Lq + UNIT_ROWS - 1) / UNIT_ROWS;
    const int nkv_all = (a.Lk + BKV - 1) / BKV;
    const int64_t units = static_cast<int64_t>(nqb) * a.BH;
    const int64_t G = std::max<int64_t>(
        1, std::min<int64_t>(std::max(ctx.num_sms, 1), units * nkv_all / MIN_RANGE));
    // a workspace slot and flags per CTA when some range starts inside a unit
    const int64_t T = (units - dp_waves(units, G) * G) * nkv_all;
    bool split = false;
    for (int64_t c = 1; c < G && !split; ++c) split = range_start(c, T, G) % nkv_all != 0;
    float *ws = nullptr;
    unsigned *flags = nullptr;
    if (split) {
        const size_t ws_bytes = static_cast<size_t>(G) * WS_FLOATS * sizeof(float);
        const size_t flag_bytes = static_cast<size_t>(G) * FLAGS_PER_SLOT * sizeof(unsigned);
        e = scratch_alloc(ws_bytes + flag_bytes, ctx, reinterpret_cast<void **>(&ws));
        if (e != cudaSuccess) return e;
        flags = reinterpret_cast<unsigned *>(reinterpret_cast<char *>(ws) + ws_bytes);
        e = cudaMemsetAsync(flags, 0, flag_bytes, ctx.stream);
    }
    if (e == cudaSuccess) {
        // a head part waits for flags other CTAs raise: every CTA must be resident at once
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(G));
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = SMEM_BYTES;
        cfg.stream = ctx.stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, attention_kernel, tmQ, tmK, tmV, tmO, a.Lq, a.Lk, c_log2, nqb,
                               units, ws, flags, ctx.err, ctx.timeout_ns);
    }
    if (ws) {
        const cudaError_t f = scratch_free(ws, ctx);
        if (e == cudaSuccess) e = f;
    }
    return e;
}

}  // namespace qgi
