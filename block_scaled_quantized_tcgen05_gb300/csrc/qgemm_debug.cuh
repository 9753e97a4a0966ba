// qgemm_debug.cuh -- bounds checks of the debug build.
//
// Built with -DQGEMM_DEBUG (`build.build(debug=True)`, the library libqgemm_debug.so, loaded by
// the binding when QGEMM_DEBUG=1), the kernels check their own index arithmetic against the
// extents they were given before each access they compute themselves: TMA coordinates (the
// 16-byte rule for the innermost coordinate, rows inside the tensor), offsets into the repacked
// scale planes and the attention workspace, TMEM columns, and global addresses of the stores the
// kernels issue directly.  A failed check sets ERR_BOUNDS in the device error word
// (qgemm_poll_device_error) and the access is skipped: nothing traps, so the context stays usable
// and the test that reads the word can say which launch went wrong.  In the release build every
// check is the constant true and no code is generated for it.
//
// It stands in for a memory sanitizer, which this library is not run under; the tests run every
// kernel route of the debug build on small and ragged shapes and require a clean error word and
// the oracle's results.
#pragma once

#include <cstdint>

namespace qg {

// The error-word bit of a failed bounds check (beside the timeout bits of qgemm_ptx.cuh).
constexpr unsigned ERR_BOUNDS = 32u;

#ifdef QGEMM_DEBUG
__device__ __forceinline__ bool bounds_ok(unsigned *err, bool ok) {
    if (!ok) atomicOr(err, ERR_BOUNDS);
    return ok;
}
#define QG_IN_BOUNDS(err, cond) (::qg::bounds_ok((err), static_cast<bool>(cond)))
#else
#define QG_IN_BOUNDS(err, cond) (true)
#endif

// [p, p + bytes) inside [base, base + extent).
#define QG_IN_RANGE(err, p, bytes, base, extent)                                               \
    QG_IN_BOUNDS((err),                                                                        \
                 reinterpret_cast<uintptr_t>(p) >= reinterpret_cast<uintptr_t>(base) &&        \
                     reinterpret_cast<uintptr_t>(p) + static_cast<uintptr_t>(bytes) <=         \
                         reinterpret_cast<uintptr_t>(base) + static_cast<uintptr_t>(extent))

}  // namespace qg
