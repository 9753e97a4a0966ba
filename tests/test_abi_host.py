"""Host-side checks of the C ABI (no GPU): the library loads, exports every declared entry point,
and rejects bad arguments with the documented status before touching the device."""
import ctypes
import os
import re

import pytest

import block_scaled_quantized_tcgen05_gb300 as q
from block_scaled_quantized_tcgen05_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return q.load_library()


def _declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert "qgemm_mxfp8" in names and "gemm_f16" in names and len(names) >= 15
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings(lib):
    for code, name in q.STATUS_NAMES.items():
        assert q.qgemm_status_string(code) == name
    assert lib.qgemm_version() >> 16 == 1


FAKE = 0x7F0000000000      # a 16-byte aligned fake device address, never dereferenced on host


def _create(lib, dt, rows, k, data, ld, scales, lds, block=32):
    out = ctypes.c_void_p()
    st = lib.qgemm_create_tensor(ctypes.byref(out), dt, rows, k, ctypes.c_void_p(data), ld,
                                 ctypes.c_void_p(scales) if scales else None, lds, block)
    return st, out


def test_create_tensor_validation(lib):
    st, t = _create(lib, q.E4M3, 128, 256, FAKE, 256, FAKE + 65536, 8)
    assert st == 0 and t.value
    lib.qgemm_destroy_tensor(t)
    assert _create(lib, 9, 4, 32, FAKE, 32, FAKE, 1)[0] == 4                   # unknown dtype
    assert _create(lib, q.E4M3, 4, 32, FAKE, 32, FAKE, 1, block=16)[0] == 4    # block != 32
    assert _create(lib, q.E4M3, 4, 48, FAKE, 48, FAKE, 2)[0] == 2              # k % 32
    assert _create(lib, q.E4M3, -1, 32, FAKE, 32, FAKE, 1)[0] == 1             # negative
    assert _create(lib, q.E4M3, 4, 32, 0, 32, FAKE, 1)[0] == 1                 # null data
    assert _create(lib, q.E4M3, 4, 64, FAKE, 32, FAKE, 2)[0] == 1              # short stride
    assert _create(lib, q.INT8, 4, 64, FAKE, 64, 0, 2)[0] == 1                 # null scales
    assert _create(lib, q.F16, 4, 64, FAKE, 128, FAKE, 2)[0] == 4              # F16 + scales
    st, t = _create(lib, q.F16, 4, 64, FAKE, 128, 0, 0)
    assert st == 0
    lib.qgemm_destroy_tensor(t)
    lib.qgemm_destroy_tensor(None)                                             # no-op


def test_slice_moves_both_planes(lib):
    st, t = _create(lib, q.INT4, 64, 256, FAKE, 128, FAKE + (1 << 20), 8)
    assert st == 0
    out = ctypes.c_void_p()
    assert lib.qgemm_tensor_slice(t, 8, 16, 64, 128, ctypes.byref(out)) == 0
    dt, rows, k = ctypes.c_int32(), ctypes.c_int64(), ctypes.c_int64()
    data, sc = ctypes.c_void_p(), ctypes.c_void_p()
    ld, lds = ctypes.c_int64(), ctypes.c_int64()
    assert lib.qgemm_tensor_info(out, ctypes.byref(dt), ctypes.byref(rows), ctypes.byref(k),
                                 ctypes.byref(data), ctypes.byref(ld), ctypes.byref(sc),
                                 ctypes.byref(lds)) == 0
    assert (dt.value, rows.value, k.value) == (q.INT4, 16, 128)
    assert data.value == FAKE + 8 * 128 + 64 // 2              # int4: k0 / 2 bytes
    assert sc.value == FAKE + (1 << 20) + 8 * 8 + 64 // 32     # scale block k0 / 32
    assert (ld.value, lds.value) == (128, 8)
    lib.qgemm_destroy_tensor(out)
    bad = ctypes.c_void_p()
    assert lib.qgemm_tensor_slice(t, 0, 65, 0, 32, ctypes.byref(bad)) == 1   # rows out of range
    assert lib.qgemm_tensor_slice(t, 0, 8, 16, 32, ctypes.byref(bad)) == 2   # k0 % 32
    assert bad.value is None
    lib.qgemm_destroy_tensor(t)


def test_compute_calls_reject_before_launch(lib):
    """Argument errors come back as status codes without any device work (no GPU here)."""
    _, a = _create(lib, q.E4M3, 128, 256, FAKE, 256, FAKE + 65536, 8)
    _, b = _create(lib, q.E4M3, 256, 256, FAKE, 256, FAKE + 65536, 8)
    _, b2 = _create(lib, q.E4M3, 256, 128, FAKE, 128, FAKE + 65536, 4)
    _, w8 = _create(lib, q.INT8, 256, 256, FAKE, 256, FAKE + 65536, 8)
    _, misal = _create(lib, q.E4M3, 256, 256, FAKE + 8, 256, FAKE + 65536, 8)
    C = ctypes.c_void_p(FAKE + (1 << 24))
    assert lib.qgemm_mxfp8(a, b2, C, 256, None) == 1            # K mismatch
    assert lib.qgemm_mxfp8(a, w8, C, 256, None) == 4            # dtype
    assert lib.qgemm_mxfp8(a, b, C, 128, None) == 1             # ldc < N
    assert lib.qgemm_mxfp8(a, b, ctypes.c_void_p(FAKE + 1), 256, None) == 3   # C misaligned
    assert lib.qgemm_mxfp8(a, misal, C, 256, None) == 3         # data misaligned
    assert lib.qgemm_mxfp8(None, b, C, 256, None) == 1
    assert lib.gemm_f16(C, 20, C, 256, C, 256, 16, 256, 20, None) == 3        # lda % 8
    assert lib.gemm_f16(C, 256, C, 256, C, 256, -1, 256, 256, None) == 1
    assert lib.qgemm_w8_gemv(C, 256, 17, w8, C, 256, None) == 2               # M > 16
    assert lib.qgemm_w8_gemv(C, 256, 0, w8, C, 256, None) == 2                # M < 1
    assert lib.qgemm_w8_gemv(C, 256, 4, a, C, 256, None) == 4                 # not INT8
    assert lib.qgemm_w4a16(C, 256, 16, w8, C, 256, None) == 4                 # not INT4
    # empty outputs are a successful no-op before any CUDA call
    _, e0 = _create(lib, q.E4M3, 0, 256, FAKE, 256, FAKE + 65536, 8)
    assert lib.qgemm_mxfp8(e0, b, C, 256, None) == 0
    assert lib.gemm_f16(C, 256, C, 256, C, 256, 0, 256, 256, None) == 0
    for t in (a, b, b2, w8, misal, e0):
        lib.qgemm_destroy_tensor(t)


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    """With the shared library missing the binding raises instead of computing anything."""
    monkeypatch.setattr(q, "_lib", None)
    monkeypatch.setattr(q, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        q.load_library()


def test_epilogue_descriptor_validation(lib):
    """The _ex calls check their epilogue descriptor (fields 0 or 1) and then every argument
    the plain call checks, all before any device work."""
    _, a = _create(lib, q.E4M3, 128, 256, FAKE, 256, FAKE + 65536, 8)
    _, b = _create(lib, q.E4M3, 256, 256, FAKE, 256, FAKE + 65536, 8)
    _, b2 = _create(lib, q.E4M3, 256, 128, FAKE, 128, FAKE + 65536, 4)
    _, w4 = _create(lib, q.INT4, 256, 256, FAKE, 128, FAKE + 65536, 8)
    _, e0 = _create(lib, q.E4M3, 0, 256, FAKE, 256, FAKE + 65536, 8)
    C = ctypes.c_void_p(FAKE + (1 << 24))
    ok = ctypes.byref(q.Epilogue(1, 1))
    assert lib.qgemm_mxfp8_ex(a, b, C, 256, ctypes.byref(q.Epilogue(2, 0)), None) == 1
    assert lib.gemm_f16_ex(C, 256, C, 256, C, 256, 16, 256, 256,
                           ctypes.byref(q.Epilogue(0, -1)), None) == 1
    assert lib.qgemm_w4a16_ex(C, 256, 16, w4, C, 256, ctypes.byref(q.Epilogue(3, 1)), None) == 1
    assert lib.qgemm_w8_gemv_ex(C, 256, 4, w4, C, 256, ok, None) == 4         # not INT8
    assert lib.qgemm_mxfp8_ex(a, b2, C, 256, ok, None) == 1                     # K mismatch
    assert lib.gemm_f16_ex(C, 20, C, 256, C, 256, 16, 256, 20, ok, None) == 3   # lda % 8
    assert lib.qgemm_mxfp8_ex(e0, b, C, 256, ok, None) == 0                     # empty output
    for t in (a, b, b2, w4, e0):
        lib.qgemm_destroy_tensor(t)


def test_mxfp4_rejects_before_launch(lib):
    """qgemm_mxfp4 and its _ex form check dtype, K, output and alignment with no device work."""
    _, a = _create(lib, q.E2M1, 128, 256, FAKE, 128, FAKE + 65536, 8)
    _, b = _create(lib, q.E2M1, 256, 256, FAKE, 128, FAKE + 65536, 8)
    _, b2 = _create(lib, q.E2M1, 256, 128, FAKE, 64, FAKE + 65536, 4)
    _, f8 = _create(lib, q.E4M3, 256, 256, FAKE, 256, FAKE + 65536, 8)
    _, misal = _create(lib, q.E2M1, 256, 256, FAKE + 8, 128, FAKE + 65536, 8)
    _, odd = _create(lib, q.E2M1, 256, 256, FAKE, 136, FAKE + 65536, 8)
    _, e0 = _create(lib, q.E2M1, 0, 256, FAKE, 128, FAKE + 65536, 8)
    C = ctypes.c_void_p(FAKE + (1 << 24))
    assert lib.qgemm_mxfp4(a, b2, C, 256, None) == 1            # K mismatch
    assert lib.qgemm_mxfp4(a, f8, C, 256, None) == 4            # E4M3 operand
    assert lib.qgemm_mxfp8(a, b, C, 256, None) == 4             # E2M1 views to the FP8 call
    assert lib.qgemm_mxfp4(a, b, C, 128, None) == 1             # ldc < N
    assert lib.qgemm_mxfp4(a, b, ctypes.c_void_p(FAKE + 1), 256, None) == 3   # C misaligned
    assert lib.qgemm_mxfp4(a, misal, C, 256, None) == 3         # data misaligned
    assert lib.qgemm_mxfp4(a, odd, C, 256, None) == 3           # row stride % 16
    assert lib.qgemm_mxfp4(None, b, C, 256, None) == 1
    assert lib.qgemm_mxfp4(e0, b, C, 256, None) == 0            # empty output: no-op
    assert lib.qgemm_mxfp4_ex(a, b, C, 256, ctypes.byref(q.Epilogue(0, 2)), None) == 1
    assert lib.qgemm_mxfp4_ex(a, f8, C, 256, ctypes.byref(q.Epilogue(1, 0)), None) == 4
    # an E2M1 view is two elements per byte: k = 256 needs 128-byte rows
    assert _create(lib, q.E2M1, 4, 256, FAKE, 100, FAKE, 8)[0] == 1
    for t in (a, b, b2, f8, misal, odd, e0):
        lib.qgemm_destroy_tensor(t)


def test_w4a16_f16s_rejects_before_launch(lib):
    """The fp16-scale int4 GEMM validates shape, strides and alignment with no device work."""
    P = ctypes.c_void_p
    A, W, S, C = (P(FAKE + off) for off in (0, 1 << 20, 1 << 22, 1 << 24))
    ok = dict(lda=256, M=16, ldw=128, lds=8, N=64, K=256, ldc=64)

    def call(A=A, W=W, S=S, C=C, **kw):
        a = dict(ok, **kw)
        return lib.qgemm_w4a16_f16s(A, a["lda"], a["M"], W, a["ldw"], S, a["lds"], a["N"],
                                    a["K"], C, a["ldc"], None)
    assert call(K=288, lda=288, ldw=144, lds=16) == 2          # K % 256
    assert call(lda=128) == 1                                  # lda < K
    assert call(ldw=64) == 1                                   # ldw < K/2
    assert call(lds=4) == 1                                    # lds < K/32
    assert call(lda=260) == 3                                  # lda % 8
    assert call(A=P(FAKE + 8)) == 3                            # A misaligned
    assert call(W=P(FAKE + (1 << 20) + 8)) == 3                # W misaligned
    assert call(ldw=136) == 3                                  # ldw % 16
    assert call(S=P(FAKE + (1 << 22) + 2)) == 3                # scales misaligned
    assert call(lds=12) == 3                                   # lds % 8
    assert call(ldc=32) == 1                                   # ldc < N
    assert call(M=-1) == 1
    assert call(M=0) == 0 and call(N=0) == 0                   # empty output: no-op
    assert lib.qgemm_w4a16_f16s_ex(A, 256, 16, W, 128, S, 8, 64, 256, C, 64,
                                   ctypes.byref(q.Epilogue(0, 5)), None) == 1


def test_mxfp8_host_rejects_before_any_cuda_call(lib):
    """qgemm_mxfp8_host validates its views and output before it touches CUDA (no GPU here)."""
    _, a = _create(lib, q.E4M3, 128, 256, FAKE, 256, FAKE + 65536, 8)
    _, b2 = _create(lib, q.E4M3, 256, 128, FAKE, 128, FAKE + 65536, 4)
    _, b = _create(lib, q.E4M3, 256, 256, FAKE, 256, FAKE + 65536, 8)
    _, w8 = _create(lib, q.INT8, 256, 256, FAKE, 256, FAKE + 65536, 8)
    C = ctypes.c_void_p(FAKE + (1 << 24))
    assert lib.qgemm_mxfp8_host(a, b2, C, 256, None) == 1      # K mismatch
    assert lib.qgemm_mxfp8_host(a, w8, C, 256, None) == 4      # dtype
    assert lib.qgemm_mxfp8_host(a, b, C, 128, None) == 1       # ldc < N
    assert lib.qgemm_mxfp8_host(a, b, None, 256, None) == 1    # no output
    _, e0 = _create(lib, q.E4M3, 0, 256, FAKE, 256, FAKE + 65536, 8)
    assert lib.qgemm_mxfp8_host(e0, b, C, 256, None) == 0      # empty output: nothing to do
    for t in (a, b2, b, w8, e0):
        lib.qgemm_destroy_tensor(t)


def test_clock_probe_argument_checks(lib):
    # rejected before anything reaches a device
    assert lib.qgemm_sm_clock_probe(100000, None, None) == 1                     # null out
    assert lib.qgemm_sm_clock_probe(0, ctypes.c_void_p(FAKE), None) == 1         # empty window
    assert lib.qgemm_sm_clock_probe(2 * 10 ** 9, ctypes.c_void_p(FAKE), None) == 1   # > 1 s
    assert lib.qgemm_sm_clock_probe(100000, ctypes.c_void_p(FAKE + 4), None) == 3    # alignment
