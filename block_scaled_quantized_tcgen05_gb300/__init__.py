"""Python binding of the block-scaled quantized GEMM library (``libqgemm.so``, C ABI).

Argument marshalling only: every function here passes torch tensors' device pointers, strides
and the current CUDA stream to the C entry point of the same name and raises ``QGemmError`` on a
non-OK status.  All arithmetic runs in the library's CUDA kernels; there is no CPU fallback, and
loading fails loudly when the library has not been built (``python -m
block_scaled_quantized_tcgen05_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

__all__ = [
    "QGemmError", "QTensor", "F16", "E4M3", "INT8", "INT4", "E2M1", "load_library", "library_path",
    "qgemm_version", "qgemm_debug_build", "qgemm_create_tensor", "qgemm_tensor_slice", "qgemm_destroy_tensor",
    "qgemm_mxfp8", "qgemm_mxfp8_scratch_bytes", "qgemm_mxfp8_host", "qgemm_mxfp4", "gemm_f16", "qgemm_w4a16", "qgemm_w4a16_f16s", "qgemm_attention", "qgemm_w8_gemv", "qgemm_dequant_debug",
    "qgemm_status_string", "qgemm_poll_device_error", "qgemm_set_wait_timeout_ns",
    "qgemm_selftest_wait_timeout", "qgemm_sm_clock_probe",
]

F16, E4M3, INT8, INT4, E2M1 = 0, 1, 2, 3, 4
OK = 0
STATUS_NAMES = {0: "QGEMM_OK", 1: "QGEMM_ERR_INVALID_ARG", 2: "QGEMM_ERR_UNSUPPORTED_SHAPE",
                3: "QGEMM_ERR_MISALIGNED", 4: "QGEMM_ERR_UNSUPPORTED_DTYPE", 5: "QGEMM_ERR_CUDA",
                6: "QGEMM_ERR_TIMEOUT"}

_lib = None


class Epilogue(ctypes.Structure):
    """qgemm_epilogue: C = relu?(A*B [+ C_old]), one fp16 rounding."""
    _fields_ = [("accumulate", ctypes.c_int32), ("relu", ctypes.c_int32)]


class QGemmError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{where}: {self.name}: {message}")


def debug_build_selected() -> bool:
    """QGEMM_DEBUG=1 selects the bounds-checking build libqgemm_debug.so (see build.py)."""
    return os.environ.get("QGEMM_DEBUG", "") == "1"


def library_path() -> str:
    return _build.DEBUG_LIB_PATH if debug_build_selected() else _build.LIB_PATH


def load_library():
    """Load libqgemm.so (built in-tree).  Raises if it is missing: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(f"{os.path.basename(path)} not built at {path}; run "
                          "`python -m block_scaled_quantized_tcgen05_gb300.build"
                          + (" --debug`" if debug_build_selected() else "`"))
    lib = ctypes.CDLL(path)
    P, I64, I32, U64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64
    S = ctypes.c_int
    sig = {
        "qgemm_version": (I32, []),
        "qgemm_debug_build": (I32, []),
        "qgemm_create_tensor": (S, [ctypes.POINTER(P), S, I64, I64, P, I64, P, I64, I32]),
        "qgemm_tensor_slice": (S, [P, I64, I64, I64, I64, ctypes.POINTER(P)]),
        "qgemm_destroy_tensor": (None, [P]),
        "qgemm_tensor_info": (S, [P, ctypes.POINTER(I32), ctypes.POINTER(I64),
                                  ctypes.POINTER(I64), ctypes.POINTER(P), ctypes.POINTER(I64),
                                  ctypes.POINTER(P), ctypes.POINTER(I64)]),
        "qgemm_mxfp8": (S, [P, P, P, I64, P]),
        "qgemm_mxfp8_noalloc": (S, [P, P, P, I64, P]),
        "qgemm_mxfp8_scratch_bytes": (S, [P, P, ctypes.POINTER(I64)]),
        "qgemm_mxfp8_ex": (S, [P, P, P, I64, ctypes.POINTER(Epilogue), P]),
        "qgemm_mxfp4": (S, [P, P, P, I64, P]),
        "qgemm_mxfp8_host": (S, [P, P, P, I64, P]),
        "qgemm_attention_f16": (S, [P, P, P, P] + [I64] * 12 + [ctypes.c_float, P]),
        "qgemm_w4a16_f16s": (S, [P, I64, I64, P, I64, P, I64, I64, I64, P, I64, P]),
        "qgemm_w4a16_f16s_ex": (S, [P, I64, I64, P, I64, P, I64, I64, I64, P, I64,
                                    ctypes.POINTER(Epilogue), P]),
        "qgemm_mxfp4_ex": (S, [P, P, P, I64, ctypes.POINTER(Epilogue), P]),
        "gemm_f16_ex": (S, [P, I64, P, I64, P, I64, I64, I64, I64, ctypes.POINTER(Epilogue), P]),
        "qgemm_w4a16_ex": (S, [P, I64, I64, P, P, I64, ctypes.POINTER(Epilogue), P]),
        "qgemm_w8_gemv_ex": (S, [P, I64, I64, P, P, I64, ctypes.POINTER(Epilogue), P]),
        "gemm_f16": (S, [P, I64, P, I64, P, I64, I64, I64, I64, P]),
        "qgemm_w4a16": (S, [P, I64, I64, P, P, I64, P]),
        "qgemm_w8_gemv": (S, [P, I64, I64, P, P, I64, P]),
        "qgemm_dequant_debug": (S, [P, P, P]),
        "qgemm_status_string": (ctypes.c_char_p, [S]),
        "qgemm_last_error_message": (ctypes.c_char_p, []),
        "qgemm_poll_device_error": (S, [P, ctypes.POINTER(ctypes.c_uint32)]),
        "qgemm_set_wait_timeout_ns": (None, [U64]),
        "qgemm_selftest_wait_timeout": (S, [U64, P]),
        "qgemm_sm_clock_probe": (S, [U64, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != OK:
        msg = load_library().qgemm_last_error_message().decode(errors="replace")
        raise QGemmError(status, where, msg)


def _stream(stream):
    """cudaStream_t of a torch.cuda.Stream (default: torch's current stream)."""
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _row_stride_bytes(t) -> int:
    if t.dim() != 2:
        raise ValueError("expected a 2-D tensor")
    if t.stride(1) != 1:
        raise ValueError("inner dimension must be contiguous")
    return t.stride(0) * t.element_size()


def _ld(t) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("expected a 2-D row-major tensor with a contiguous inner dimension")
    return t.stride(0)


class QTensor:
    """Owning Python handle of a qgemm_tensor view; keeps the borrowed torch tensors alive."""

    def __init__(self, handle: int, dtype: int, rows: int, k: int, refs):
        self.handle = ctypes.c_void_p(handle)
        self.dtype, self.rows, self.k = dtype, rows, k
        self._refs = refs

    def close(self):
        if self.handle and self.handle.value:
            load_library().qgemm_destroy_tensor(self.handle)
            self.handle = ctypes.c_void_p(None)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def qgemm_version() -> int:
    return load_library().qgemm_version()


def qgemm_debug_build() -> bool:
    """True when the loaded library is the bounds-checking debug build."""
    return load_library().qgemm_debug_build() == 1


def qgemm_status_string(status: int) -> str:
    return load_library().qgemm_status_string(status).decode()


def qgemm_create_tensor(dtype: int, data, scales=None, rows: int | None = None,
                        k: int | None = None, block_k: int = 32) -> QTensor:
    """View of a [rows, k] quantized matrix.  ``data`` is a 2-D device tensor holding the data
    plane row-major (uint8 for E4M3 / INT8 / packed INT4 or E2M1, fp16 for F16); ``scales`` is the
    [rows, k/32] uint8 UE8M0 plane (None for F16)."""
    lib = load_library()
    rows = data.shape[0] if rows is None else rows
    if k is None:
        k = {F16: data.shape[1], E4M3: data.shape[1], INT8: data.shape[1],
             INT4: 2 * data.shape[1], E2M1: 2 * data.shape[1]}[dtype]
    out = ctypes.c_void_p()
    st = lib.qgemm_create_tensor(ctypes.byref(out), dtype, rows, k, _ptr(data),
                                 _row_stride_bytes(data), _ptr(scales),
                                 _row_stride_bytes(scales) if scales is not None else 0, block_k)
    _check(st, "qgemm_create_tensor")
    return QTensor(out.value, dtype, rows, k, (data, scales))


def qgemm_tensor_slice(t: QTensor, row0: int, nrows: int, k0: int, nk: int) -> QTensor:
    lib = load_library()
    out = ctypes.c_void_p()
    _check(lib.qgemm_tensor_slice(t.handle, row0, nrows, k0, nk, ctypes.byref(out)),
           "qgemm_tensor_slice")
    return QTensor(out.value, t.dtype, nrows, nk, t._refs)


def qgemm_destroy_tensor(t: QTensor):
    t.close()


def qgemm_mxfp8(A: QTensor, B: QTensor, C, stream=None):
    _check(load_library().qgemm_mxfp8(A.handle, B.handle, _ptr(C), _ld(C), _stream(stream)),
           "qgemm_mxfp8")
    return C


def qgemm_mxfp4(A: QTensor, B: QTensor, C, stream=None):
    """C = A B^T with E2M1 operands (UE8M0 scale per 32 along K), fp32 accumulation, fp16 out."""
    _check(load_library().qgemm_mxfp4(A.handle, B.handle, _ptr(C), _ld(C), _stream(stream)),
           "qgemm_mxfp4")
    return C


def qgemm_mxfp8_host(A: QTensor, B: QTensor, C, stream=None):
    """qgemm_mxfp8 with A, B (views of host tensors, preferably pinned) and C (a host fp16 tensor)
    in host memory: uploads, computes and downloads with the three overlapped; asynchronous on
    ``stream`` (synchronise it before reading C)."""
    if C.is_cuda:
        raise ValueError("C must be a host tensor")
    _check(load_library().qgemm_mxfp8_host(A.handle, B.handle, _ptr(C), _ld(C), _stream(stream)),
           "qgemm_mxfp8_host")
    return C


def qgemm_mxfp8_scratch_bytes(A: QTensor, B: QTensor) -> int:
    """Bytes of pooled device scratch one qgemm_mxfp8 call on these views takes (0: none)."""
    n = ctypes.c_int64(0)
    _check(load_library().qgemm_mxfp8_scratch_bytes(A.handle, B.handle, ctypes.byref(n)),
           "qgemm_mxfp8_scratch_bytes")
    return n.value


def qgemm_mxfp8_noalloc(A: QTensor, B: QTensor, C, stream=None):
    """qgemm_mxfp8 with its scale scratch in the library's fixed device buffer: allocates no
    device memory (for callers that cannot allocate mid-run); shapes needing more than 8 MiB of
    repacked scales are rejected; concurrent calls on one device must not overlap on the GPU."""
    _check(load_library().qgemm_mxfp8_noalloc(A.handle, B.handle, _ptr(C), _ld(C),
                                               _stream(stream)), "qgemm_mxfp8_noalloc")
    return C


def gemm_f16(A, B, C, stream=None):
    M, K = A.shape
    N = B.shape[1]
    _check(load_library().gemm_f16(_ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C), _ld(C), M, N, K,
                                   _stream(stream)), "gemm_f16")
    return C


def qgemm_w4a16(A, W: QTensor, C, stream=None):
    _check(load_library().qgemm_w4a16(_ptr(A), _ld(A), A.shape[0], W.handle, _ptr(C), _ld(C),
                                      _stream(stream)), "qgemm_w4a16")
    return C


def qgemm_w8_gemv(X, W: QTensor, Y, stream=None):
    _check(load_library().qgemm_w8_gemv(_ptr(X), _ld(X), X.shape[0], W.handle, _ptr(Y), _ld(Y),
                                        _stream(stream)), "qgemm_w8_gemv")
    return Y


def _epi(accumulate: bool, relu: bool):
    return ctypes.byref(Epilogue(int(bool(accumulate)), int(bool(relu))))


def qgemm_mxfp8_ex(A: QTensor, B: QTensor, C, accumulate=False, relu=False, stream=None):
    """C = relu?(A B^T [+ C]) with the MXFP8 operands of qgemm_mxfp8."""
    _check(load_library().qgemm_mxfp8_ex(A.handle, B.handle, _ptr(C), _ld(C),
                                         _epi(accumulate, relu), _stream(stream)), "qgemm_mxfp8_ex")
    return C


def qgemm_mxfp4_ex(A: QTensor, B: QTensor, C, accumulate=False, relu=False, stream=None):
    """C = relu?(A B^T [+ C]) with the MXFP4 operands of qgemm_mxfp4."""
    _check(load_library().qgemm_mxfp4_ex(A.handle, B.handle, _ptr(C), _ld(C),
                                         _epi(accumulate, relu), _stream(stream)), "qgemm_mxfp4_ex")
    return C


def gemm_f16_ex(A, B, C, accumulate=False, relu=False, stream=None):
    M, K = A.shape
    N = B.shape[1]
    _check(load_library().gemm_f16_ex(_ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C), _ld(C), M, N, K,
                                      _epi(accumulate, relu), _stream(stream)), "gemm_f16_ex")
    return C


def qgemm_w4a16_ex(A, W: QTensor, C, accumulate=False, relu=False, stream=None):
    _check(load_library().qgemm_w4a16_ex(_ptr(A), _ld(A), A.shape[0], W.handle, _ptr(C), _ld(C),
                                         _epi(accumulate, relu), _stream(stream)), "qgemm_w4a16_ex")
    return C


def qgemm_attention(Q, K, V, O, scale=None, stream=None):
    """O = softmax(scale Q K^T) V per head; Q, O [BH, Lq, 128], K, V [BH, Lk, 128] fp16 device
    tensors with a contiguous last dimension; scale defaults to 1/sqrt(128)."""
    for t in (Q, K, V, O):
        if t.dim() != 3 or t.stride(2) != 1:
            raise ValueError("expected [BH, L, d] tensors with a contiguous last dimension")
    BH, Lq, d = Q.shape
    Lk = K.shape[1]
    if scale is None:
        scale = d ** -0.5
    _check(load_library().qgemm_attention_f16(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(O), BH, Lq, Lk, d, Q.stride(0), Q.stride(1),
        K.stride(0), K.stride(1), V.stride(0), V.stride(1), O.stride(0), O.stride(1),
        float(scale), _stream(stream)), "qgemm_attention_f16")
    return O


def qgemm_w4a16_f16s(A, W, S, C, stream=None):
    """C = A W^T with int4 W [N, K/2] (packed uint8) and fp16 block-32 scales S [N, K/32], each
    weight dequantised to the half nearest q * s (the custom-format escape hatch)."""
    M, K = A.shape
    N = W.shape[0]
    _check(load_library().qgemm_w4a16_f16s(_ptr(A), _ld(A), M, _ptr(W), _row_stride_bytes(W),
                                           _ptr(S), _ld(S), N, K, _ptr(C), _ld(C),
                                           _stream(stream)), "qgemm_w4a16_f16s")
    return C


def qgemm_w4a16_f16s_ex(A, W, S, C, accumulate=False, relu=False, stream=None):
    M, K = A.shape
    N = W.shape[0]
    _check(load_library().qgemm_w4a16_f16s_ex(_ptr(A), _ld(A), M, _ptr(W), _row_stride_bytes(W),
                                              _ptr(S), _ld(S), N, K, _ptr(C), _ld(C),
                                              _epi(accumulate, relu), _stream(stream)),
           "qgemm_w4a16_f16s_ex")
    return C


def qgemm_w8_gemv_ex(X, W: QTensor, Y, accumulate=False, relu=False, stream=None):
    _check(load_library().qgemm_w8_gemv_ex(_ptr(X), _ld(X), X.shape[0], W.handle, _ptr(Y), _ld(Y),
                                           _epi(accumulate, relu), _stream(stream)),
           "qgemm_w8_gemv_ex")
    return Y


def qgemm_dequant_debug(t: QTensor, out, stream=None):
    _check(load_library().qgemm_dequant_debug(t.handle, _ptr(out), _stream(stream)),
           "qgemm_dequant_debug")
    return out


def qgemm_poll_device_error(stream=None) -> int:
    """Synchronise and return (and clear) the device error word; 0 when no wait gave up."""
    code = ctypes.c_uint32(0)
    st = load_library().qgemm_poll_device_error(_stream(stream), ctypes.byref(code))
    if st not in (OK, 6):
        _check(st, "qgemm_poll_device_error")
    return code.value


def qgemm_set_wait_timeout_ns(ns: int):
    load_library().qgemm_set_wait_timeout_ns(int(ns))


def qgemm_selftest_wait_timeout(timeout_ns: int, stream=None):
    _check(load_library().qgemm_selftest_wait_timeout(int(timeout_ns), _stream(stream)),
           "qgemm_selftest_wait_timeout")


def qgemm_sm_clock_probe(window_ns: int, out, stream=None):
    """Write (SM cycles, global-timer ns) over `window_ns` into the two int64 elements of the
    device tensor `out` (from the GPU, on `stream`)."""
    _check(load_library().qgemm_sm_clock_probe(int(window_ns), _ptr(out), _stream(stream)),
           "qgemm_sm_clock_probe")
