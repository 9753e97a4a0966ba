"""CPU oracle for the block-scaled quantized matmul.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg are the only callers.  The library's product path never imports this package,
and this package never imports the library.  The arithmetic lives in ``qgemm_oracle.c`` (plain C,
fp64); this module only compiles it with gcc and marshals numpy arrays through ctypes.

Functions and the passages they follow:

* ``e4m3_table`` / ``ue8m0_table`` -- decode of every code of the data type (FP8 E4M3, "Optimize
  custom machine learning operations with Metal tensors", section "Shader MXFP8 tensor types")
  and of the block scale type (UE8M0 = FP8 E8M0, "TensorOps: quantized matmul, cooperative
  tensors, and the neural accelerator", section "Kernel-phase findings", fact 2).
* ``dequant`` -- element times the scale of its 32-element block along K ("TensorOps: quantized
  matmul ...", section "Scale planes: one MTLTensor = data + scales"); int4 nibble order from the
  same page, section "VALIDATED ON M4 MAX", fact 5.
* ``dequant_int4_f16s`` / ``w4a16_f16s`` -- the custom-format escape hatch: int4 weights with
  arbitrary fp16 scales per block of 32 along K ("TensorOps: quantized matmul ...", sections
  "Revised kernel strategy" and "M2 = block-32 fp16 scaling"), each weight dequantised to
  fp16_rn(q * s) as that recipe's half multiply gives, then the product over those weights.
* ``attention`` -- fused attention ("TensorOps: quantized matmul ...", section "FlashAttention on
  TensorOps (the recipe)"; "Optimize custom machine learning operations with Metal tensors",
  section on FlashAttention with cooperative tensors): Q K^T scaled, each row's maximum, exp of
  the scores minus it, normalised by the row sum, times V, all in fp64.
* ``mxfp8`` / ``gemm_f16`` / ``w4a16`` / ``w8_gemv`` -- C = A * B^T over the decoded operands in
  fp64 (matmul2d, mode multiply: "TensorOps: quantized matmul ...", section "The real matmul2d
  API"), reported as IEEE binary16 round-to-nearest-even.

Every function returns the exact-in-fp64 product ``C``, the magnitude sum ``D = sum |a*b|`` that
the tolerance is normalised by, and the fp16 bits of ``C``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qgemm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

# dtype codes of qgemm_oracle.c
F16, E4M3, INT8, INT4, E2M1 = 0, 1, 2, 3, 4

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile qgemm_oracle.c with gcc (OpenMP, no fp contraction, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        lib.orc_e4m3.restype = ctypes.c_double
        lib.orc_e4m3.argtypes = [ctypes.c_uint8]
        lib.orc_ue8m0.restype = ctypes.c_double
        lib.orc_ue8m0.argtypes = [ctypes.c_uint8]
        lib.orc_f16.restype = ctypes.c_double
        lib.orc_f16.argtypes = [ctypes.c_uint16]
        lib.orc_f16_rn.restype = ctypes.c_uint16
        lib.orc_f16_rn.argtypes = [ctypes.c_double]
        lib.orc_int4_get.restype = I
        lib.orc_int4_get.argtypes = [P, I64]
        lib.orc_int8_get.restype = I
        lib.orc_int8_get.argtypes = [ctypes.c_uint8]
        lib.orc_dequant.restype = None
        lib.orc_dequant.argtypes = [I, I64, I64, P, I64, P, I64, P, P]
        lib.orc_dequant_int4_f16s.restype = None
        lib.orc_dequant_int4_f16s.argtypes = [I64, I64, P, I64, P, I64, P, P]
        lib.orc_attention.restype = None
        lib.orc_attention.argtypes = [I64, P, P, I64, I64, P, I64, I64, P, I64, I64, P, I64, I64,
                                      ctypes.c_double, P, P]
        lib.orc_dequant_f16_kn.restype = None
        lib.orc_dequant_f16_kn.argtypes = [I64, I64, P, I64, P, P]
        lib.orc_dot_rows.restype = None
        lib.orc_dot_rows.argtypes = [I64, I64, I64, P, P, P, P]
        lib.orc_dot_quant.restype = None
        lib.orc_dot_quant.argtypes = [I64, I64, I64, P, I, P, I64, P, I64, P, P]
        lib.orc_f16_rn_array.restype = None
        lib.orc_f16_rn_array.argtypes = [I64, P, P]
        lib.orc_e2m1.restype = ctypes.c_double
        lib.orc_e2m1.argtypes = [ctypes.c_uint8]
        lib.orc_e2m1_table.restype = None
        lib.orc_e2m1_table.argtypes = [P]
        lib.orc_e4m3_table.restype = None
        lib.orc_e4m3_table.argtypes = [P]
        lib.orc_ue8m0_table.restype = None
        lib.orc_ue8m0_table.argtypes = [P]
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u8(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.uint8:
        a = a.view(np.uint8)
    return np.ascontiguousarray(a)


# ----------------------------------------------------------------------------- decoders
def e2m1_table() -> np.ndarray:
    """Values of the 16 E2M1 codes (low nibble), fp64."""
    out = np.empty(16, np.float64)
    _load().orc_e2m1_table(_ptr(out))
    return out


def e4m3_table() -> np.ndarray:
    out = np.empty(256, np.float64)
    _load().orc_e4m3_table(_ptr(out))
    return out


def ue8m0_table() -> np.ndarray:
    out = np.empty(256, np.float64)
    _load().orc_ue8m0_table(_ptr(out))
    return out


def f16_value(bits: int) -> float:
    return _load().orc_f16(int(bits))


def f16_rn(x) -> np.ndarray:
    """fp16 bits (uint16) of round-to-nearest-even of each fp64 value."""
    x = np.ascontiguousarray(np.asarray(x, np.float64))
    out = np.empty(x.shape, np.uint16)
    _load().orc_f16_rn_array(x.size, _ptr(x), _ptr(out))
    return out


def int4_get(packed_row: np.ndarray, k: int) -> int:
    row = _u8(packed_row)
    return _load().orc_int4_get(_ptr(row), int(k))


def dequant(dtype: int, data, scales, rows: np.ndarray | None = None, k: int | None = None
            ) -> np.ndarray:
    """Decoded fp64 [len(rows), k] of a quantized plane.

    ``data`` is [R, bytes_per_row] uint8 (or int8/fp16 viewed as bytes); ``scales`` is
    [R, k/32] uint8 (ignored for F16).  ``rows`` selects rows (default all)."""
    d = _u8(data)
    if d.ndim != 2:
        raise ValueError("data must be 2-D")
    R = d.shape[0]
    if k is None:
        k = {F16: d.shape[1] // 2, E4M3: d.shape[1], INT8: d.shape[1], INT4: d.shape[1] * 2,
             E2M1: d.shape[1] * 2}[dtype]
    s = _u8(scales) if scales is not None else np.zeros((R, 1), np.uint8)
    idx = None if rows is None else np.ascontiguousarray(np.asarray(rows, np.int64))
    n = R if idx is None else idx.size
    out = np.empty((n, k), np.float64)
    _load().orc_dequant(dtype, n, k, _ptr(d), d.shape[1], _ptr(s), s.shape[1], _ptr(idx),
                        _ptr(out))
    return out


def dequant_int4_f16s(w_packed, s_f16, rows: np.ndarray | None = None) -> np.ndarray:
    """fp64 [len(rows), K] of int4 weights [R, K/2] with fp16 scales [R, K/32]: each element is
    the fp16 value nearest (ties to even) to int4 * scale."""
    d = _u8(w_packed)
    sc = np.ascontiguousarray(np.asarray(s_f16).view(np.uint16))
    R, k = d.shape[0], d.shape[1] * 2
    if sc.shape != (R, k // 32):
        raise ValueError("scales must be [rows, K/32] fp16")
    idx = None if rows is None else np.ascontiguousarray(np.asarray(rows, np.int64))
    n = R if idx is None else idx.size
    out = np.empty((n, k), np.float64)
    _load().orc_dequant_int4_f16s(n, k, _ptr(d), d.shape[1], _ptr(sc), sc.shape[1], _ptr(idx),
                                  _ptr(out))
    return out


def dequant_f16_kn(b, cols: np.ndarray | None = None) -> np.ndarray:
    """fp16 [K, N] row-major -> fp64 [len(cols), K] (the transposed right operand)."""
    b = np.ascontiguousarray(np.asarray(b).view(np.uint16))
    K, N = b.shape
    idx = None if cols is None else np.ascontiguousarray(np.asarray(cols, np.int64))
    n = N if idx is None else idx.size
    out = np.empty((n, K), np.float64)
    _load().orc_dequant_f16_kn(n, K, _ptr(b), N, _ptr(idx), _ptr(out))
    return out


def dot_rows(A: np.ndarray, B: np.ndarray):
    """C = A @ B.T and D = |A| @ |B|.T by plain fp64 loops."""
    A = np.ascontiguousarray(A, np.float64)
    B = np.ascontiguousarray(B, np.float64)
    assert A.shape[1] == B.shape[1]
    C = np.empty((A.shape[0], B.shape[0]), np.float64)
    D = np.empty_like(C)
    _load().orc_dot_rows(A.shape[0], B.shape[0], A.shape[1], _ptr(A), _ptr(B), _ptr(C), _ptr(D))
    return C, D


class Result:
    """Oracle output for a set of rows of C: exact product, magnitude sum, fp16 bits."""

    def __init__(self, C: np.ndarray, D: np.ndarray, rows: np.ndarray | None):
        self.C = C
        self.D = D
        self.rows = rows
        self.f16_bits = f16_rn(C)

    @property
    def f16(self) -> np.ndarray:
        return self.f16_bits.view(np.float16)


# ------------------------------------------------------------------------- the products
def mxfp8(a, sa, b, sb, rows=None) -> Result:
    """C[m,n] = sum_k e4m3(A[m,k]) 2^(SA[m,k/32]-127) * e4m3(B[n,k]) 2^(SB[n,k/32]-127).

    A is [M,K] E4M3 bytes, B is [N,K] E4M3 bytes (K contiguous), scales [rows, K/32] UE8M0."""
    K = _u8(a).shape[1]
    Ad = dequant(E4M3, a, sa, rows, K)
    Bd = dequant(E4M3, b, sb, None, K)
    C, D = dot_rows(Ad, Bd)
    return Result(C, D, rows)


def mxfp4(a, sa, b, sb, k=None, rows=None) -> Result:
    """C[m,n] = sum_k e2m1(A[m,k]) 2^(SA[m,k/32]-127) * e2m1(B[n,k]) 2^(SB[n,k/32]-127).

    A is [M,K/2] and B [N,K/2] packed E2M1 bytes (even k in the low nibble), scales
    [rows, K/32] UE8M0."""
    K = k if k is not None else _u8(a).shape[1] * 2
    Ad = dequant(E2M1, a, sa, rows, K)
    Bd = dequant(E2M1, b, sb, None, K)
    C, D = dot_rows(Ad, Bd)
    return Result(C, D, rows)


def gemm_f16(a, b, rows=None) -> Result:
    """C = A[M,K] @ B[K,N], fp16 inputs (row-major), exact products summed in fp64."""
    a16 = np.ascontiguousarray(np.asarray(a).view(np.uint16))
    K = a16.shape[1]
    Ad = dequant(F16, a16.view(np.uint8), None, rows, K)
    Bd = dequant_f16_kn(b)
    C, D = dot_rows(Ad, Bd)
    return Result(C, D, rows)


def w4a16(a, w_packed, sw, rows=None) -> Result:
    """C[m,n] = sum_k A[m,k] * int4(W[n,k]) 2^(SW[n,k/32]-127); A fp16 [M,K], W packed [N,K/2]."""
    a16 = np.ascontiguousarray(np.asarray(a).view(np.uint16))
    K = a16.shape[1]
    Ad = dequant(F16, a16.view(np.uint8), None, rows, K)
    Wd = dequant(INT4, w_packed, sw, None, K)
    C, D = dot_rows(Ad, Wd)
    return Result(C, D, rows)


def w4a16_f16s(a, w_packed, s_f16, rows=None) -> Result:
    """C[m,n] = sum_k A[m,k] * fp16_rn(int4(W[n,k]) * S[n,k/32]); A fp16 [M,K], W packed int4
    [N,K/2], S fp16 [N,K/32] (any finite or infinite fp16 values)."""
    a16 = np.ascontiguousarray(np.asarray(a).view(np.uint16))
    K = a16.shape[1]
    Ad = dequant(F16, a16.view(np.uint8), None, rows, K)
    Wd = dequant_int4_f16s(w_packed, s_f16)
    C, D = dot_rows(Ad, Wd)
    return Result(C, D, rows)


def attention(q, k, v, scale: float, heads=None, qrows=None) -> Result:
    """O = softmax(scale * Q K^T) V per head, q [BH, Lq, d], k and v [BH, Lk, d] fp16 (numpy or
    torch CPU).  ``heads`` / ``qrows`` select output rows (default: every (head, row) pair, in
    order); the Result holds O and D as [n, d]."""
    Q = np.ascontiguousarray(np.asarray(q).view(np.uint16))
    K = np.ascontiguousarray(np.asarray(k).view(np.uint16))
    V = np.ascontiguousarray(np.asarray(v).view(np.uint16))
    BH, Lq, d = Q.shape
    Lk = K.shape[1]
    if heads is None:
        heads = np.repeat(np.arange(BH, dtype=np.int64), Lq)
        qrows = np.tile(np.arange(Lq, dtype=np.int64), BH)
    heads = np.ascontiguousarray(np.asarray(heads, np.int64))
    qrows = np.ascontiguousarray(np.asarray(qrows, np.int64))
    n = heads.size
    O = np.empty((n, d), np.float64)
    D = np.empty((n, d), np.float64)
    _load().orc_attention(n, _ptr(heads), _ptr(qrows), Lk, d, _ptr(Q), Lq * d, d, _ptr(K),
                          Lk * d, d, _ptr(V), Lk * d, d, float(scale), _ptr(O), _ptr(D))
    return Result(O, D, None)


def w8_gemv(x, w, sw) -> Result:
    """Y[m,n] = sum_k X[m,k] * int8(W[n,k]) 2^(SW[n,k/32]-127); W decoded row by row."""
    x16 = np.ascontiguousarray(np.asarray(x).view(np.uint16))
    M, K = x16.shape
    Xd = dequant(F16, x16.view(np.uint8), None, None, K)
    wb = _u8(w)
    s = _u8(sw)
    Nw = wb.shape[0]
    C = np.empty((M, Nw), np.float64)
    D = np.empty_like(C)
    _load().orc_dot_quant(M, Nw, K, _ptr(Xd), INT8, _ptr(wb), wb.shape[1], _ptr(s), s.shape[1],
                          _ptr(C), _ptr(D))
    return Result(C, D, None)


def epilogue(res: Result, c_old=None, relu: bool = False) -> Result:
    """The fused output epilogue on an exact product.

    "TensorOps: quantized matmul ..." (section "The real matmul2d API"): mode multiply_accumulate
    computes C = A*B + C.  "Running inline ML operations in a shader with Metal 4" (section
    "Combine an element-wise function"): ReLU, max(x, 0), on each product element before the
    store.  Here C' = relu?(C + C_old) in fp64, rounded once to fp16 by Result; C_old (fp16, the
    shape of res.C) is exact in fp64 and adds |C_old| to the magnitude D of the tolerance.
    ReLU of x <= 0 is +0."""
    C = np.array(res.C, np.float64, copy=True)
    D = np.array(res.D, np.float64, copy=True)
    if c_old is not None:
        old = np.asarray(c_old, np.float16).astype(np.float64)
        if old.shape != C.shape:
            raise ValueError(f"c_old shape {old.shape} != result shape {C.shape}")
        C = C + old
        D = D + np.abs(old)
    if relu:
        C = np.where(C > 0.0, C, 0.0)
    return Result(C, D, res.rows)


def dequant_plane(dtype: int, data, scales, k: int) -> np.ndarray:
    """What the dequantise-only debug kernel must reproduce: decoded fp64 values."""
    return dequant(dtype, data, scales, None, k)


def within_tolerance(got: np.ndarray, res: Result, rel: float = 2e-3,
                     rows: np.ndarray | None = None):
    """Element-wise check |got - C| <= rel * D + 2^-24 (fp16 output quantum), where C is the
    fp64 product and D = sum |a*b|.  Non-finite reference values (fp16 overflow or NaN) must be
    matched exactly; an fp32 sum that lands on the other side of the fp16 overflow threshold is
    accepted only when C is within the tolerance of that threshold.  Returns (ok, worst, info)."""
    g = np.asarray(got, np.float64)
    C, D = res.C, res.D
    if rows is not None:
        C, D = C[rows], D[rows]
    ref16 = res.f16.astype(np.float64)
    if rows is not None:
        ref16 = ref16[rows]
    bound = rel * D + 2.0 ** -24
    fin_ref = np.isfinite(ref16)
    fin_got = np.isfinite(g)
    err = np.where(fin_ref & fin_got, np.abs(g - C), 0.0)
    # overflow threshold of binary16 under round-to-nearest-even
    near_ovf = np.abs(np.abs(C) - 65520.0) <= bound
    mism = (fin_ref != fin_got) & ~near_ovf
    nan_mism = (np.isnan(ref16) != np.isnan(g))
    sign_mism = (~fin_ref & ~fin_got & ~np.isnan(ref16) & (np.sign(ref16) != np.sign(g)))
    bad = (err > bound) | mism | nan_mism | sign_mism
    ratio = np.where(bound > 0, err / bound, 0.0)
    worst = float(ratio.max()) if ratio.size else 0.0
    nz = D > 0
    rel_err = float((err[nz] / D[nz]).max()) if nz.any() else 0.0
    info = {"n_bad": int(bad.sum()), "worst_err_over_bound": worst, "max_err_over_D": rel_err}
    return (not bad.any()), worst, info


def cosine(got: np.ndarray, ref: np.ndarray) -> float:
    g = np.asarray(got, np.float64).ravel()
    r = np.asarray(ref, np.float64).ravel()
    den = np.linalg.norm(g) * np.linalg.norm(r)
    return float(g @ r / den) if den > 0 else 1.0
