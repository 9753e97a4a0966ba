"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test ties one oracle function to a library routine, a closed form, an invariant or an exact
rational brute force, so that a dropped term, a wrong sign, a swapped index or a transposed
operand in the oracle fails at least one of them.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from block_scaled_quantized_tcgen05_gb300 import synth


# ------------------------------------------------------------------------ decode tables
def test_e4m3_table_matches_torch_float8(orc):
    """All 256 E4M3 codes equal PyTorch's float8_e4m3fn -> fp64 conversion (OCP E4M3)."""
    t = orc.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(t, ref, equal_nan=True)
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.isnan(t).sum() == 2          # one NaN pattern per sign, no infinity


def test_e4m3_closed_form_points(orc):
    """Largest finite 448 = 1.75 * 2^8, smallest subnormal 2^-9, smallest normal 2^-6, 1.0."""
    t = orc.e4m3_table()
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0
    assert t[0x01] == 2.0 ** -9 and t[0x08] == 2.0 ** -6 and t[0x38] == 1.0
    assert t[0x00] == 0.0 and np.signbit(t[0x80])
    finite = t[np.isfinite(t)]
    pos = np.sort(finite[finite > 0])
    assert pos.size == 126 and np.all(np.diff(pos) > 0)     # strictly monotone codes 1..126
    assert np.array_equal(t[1:127], pos)


def test_ue8m0_table_matches_torch_e8m0(orc):
    """All 256 UE8M0 codes equal PyTorch's float8_e8m0fnu conversion: 2^(e-127), 0xFF NaN."""
    u = orc.ue8m0_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    assert np.array_equal(u, ref, equal_nan=True)
    assert u[127] == 1.0 and u[128] == 2.0 and u[0] == 2.0 ** -127 and np.isnan(u[255])
    assert np.all(u[1:255] == 2.0 * u[0:254])


# ----------------------------------------------------------------------- fp16 rounding
def test_f16_rn_matches_numpy(orc):
    """fp64 -> binary16 round-to-nearest-even agrees with numpy's float16 cast, including
    exact ties, the subnormal range and the overflow threshold."""
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.uniform(-9, 5, 20000),
        (np.arange(-3000, 3000) + 0.5) * 2.0 ** -24,           # subnormal ties
        (1024 + np.arange(0, 2048) + 0.5) * 2.0 ** -10,        # ties in [1, 3)
        np.array([65504.0, 65519.999, 65520.0, 65536.0, -65520.0, 1e9, 0.0, -0.0,
                  2.0 ** -25, 2.0 ** -25 * 1.0000001, 2.0 ** -14 - 2.0 ** -30]),
    ])
    got = orc.f16_rn(x)
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_f16_decode_all_codes(orc):
    codes = np.arange(65536, dtype=np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    got = np.array([orc.f16_value(int(c)) for c in codes[::7]])
    assert np.array_equal(got, ref[::7], equal_nan=True)


# ----------------------------------------------------------------------- integer planes
def test_int4_nibble_order_follows_page_rule(orc):
    """Packing per the page's rule byte = (v[2i] & 0xF) | ((v[2i+1] & 0xF) << 4) decodes back to
    the two's-complement values, even index from the low nibble."""
    vals = list(range(-8, 8)) + [7, -8, 0, 1, -1, 3]
    packed = np.array([(vals[2 * i] & 0xF) | ((vals[2 * i + 1] & 0xF) << 4)
                       for i in range(len(vals) // 2)], np.uint8)
    got = [orc.int4_get(packed, k) for k in range(len(vals))]
    assert got == vals
    q = torch.tensor([vals], dtype=torch.int8)
    assert np.array_equal(synth.pack_int4(q).numpy()[0], packed)


def test_int8_dequant_is_twos_complement(orc):
    data = np.arange(256, dtype=np.uint8).reshape(8, 32)
    sc = np.full((8, 1), 127, np.uint8)
    got = orc.dequant(orc.INT8, data, sc)
    assert np.array_equal(got.ravel(), data.view(np.int8).astype(np.float64).ravel())


def test_scale_maps_to_block_of_32_along_k(orc):
    """Element (r, k) takes scale S[r, k // 32]: a distinct scale per (row, block) shows it."""
    rows, K = 3, 128
    data = np.full((rows, K), 0x38, np.uint8)               # E4M3 1.0 everywhere
    sc = (np.arange(rows * (K // 32), dtype=np.uint8).reshape(rows, K // 32) + 120)
    got = orc.dequant(orc.E4M3, data, sc)
    want = np.repeat(2.0 ** (sc.astype(np.float64) - 127), 32, axis=1)
    assert np.array_equal(got, want)


# -------------------------------------------------------------------------- products
def _rand_e4m3(rng, shape):
    b = rng.integers(0, 256, shape, dtype=np.uint8)
    b[(b & 0x7F) == 0x7F] = 0x3C                          # no NaN codes
    return b


def _torch_dequant_e4m3(b, s):
    v = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    sc = torch.from_numpy(s).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    return v * np.repeat(sc, 32, axis=1)


def test_mxfp8_brute_force_exact_rationals(orc):
    """Tiny shapes: the oracle equals sum of exact rational products within fp64 rounding."""
    rng = np.random.default_rng(1)
    for (M, N, K) in [(1, 1, 32), (3, 2, 64), (4, 4, 64), (2, 3, 32)]:
        a = _rand_e4m3(rng, (M, K))
        b = _rand_e4m3(rng, (N, K))
        sa = rng.integers(110, 140, (M, K // 32), dtype=np.uint8)
        sb = rng.integers(110, 140, (N, K // 32), dtype=np.uint8)
        res = orc.mxfp8(a, sa, b, sb)
        A = _torch_dequant_e4m3(a, sa)
        B = _torch_dequant_e4m3(b, sb)
        for m in range(M):
            for n in range(N):
                exact = sum(Fraction(A[m, k]) * Fraction(B[n, k]) for k in range(K))
                mag = sum(abs(Fraction(A[m, k]) * Fraction(B[n, k])) for k in range(K))
                assert abs(Fraction(res.C[m, n]) - exact) <= Fraction(2.0 ** -50) * mag
                assert Fraction(res.D[m, n]) == pytest.approx(float(mag), rel=1e-14)
                f16 = np.float16(float(exact)).view(np.uint16)
                assert res.f16_bits[m, n] == f16 or abs(float(exact)) < 2.0 ** -20


def test_mxfp8_matches_library_matmul(orc):
    """Library special case: fp64 matmul of torch-decoded operands, non-square, 1e-12 of D."""
    rng = np.random.default_rng(2)
    M, N, K = 48, 80, 256
    a = _rand_e4m3(rng, (M, K))
    b = _rand_e4m3(rng, (N, K))
    sa = rng.integers(100, 150, (M, K // 32), dtype=np.uint8)
    sb = rng.integers(100, 150, (N, K // 32), dtype=np.uint8)
    res = orc.mxfp8(a, sa, b, sb)
    A = _torch_dequant_e4m3(a, sa)
    B = _torch_dequant_e4m3(b, sb)
    C = A @ B.T
    D = np.abs(A) @ np.abs(B).T
    assert np.all(np.abs(res.C - C) <= 1e-12 * D)
    assert np.allclose(res.D, D, rtol=1e-12)
    rows = np.array([5, 0, 47, 13])
    sub = orc.mxfp8(a, sa, b, sb, rows=rows)
    assert np.array_equal(sub.C, res.C[rows])


def test_mxfp8_invariants(orc):
    """Doubling every A scale doubles C exactly; identity and one-hot-K give closed forms."""
    rng = np.random.default_rng(3)
    M, N, K = 32, 40, 128
    a = _rand_e4m3(rng, (M, K))
    b = _rand_e4m3(rng, (N, K))
    sa = rng.integers(110, 140, (M, K // 32), dtype=np.uint8)
    sb = rng.integers(110, 140, (N, K // 32), dtype=np.uint8)
    base = orc.mxfp8(a, sa, b, sb)
    dbl = orc.mxfp8(a, sa + 1, b, sb)
    assert np.array_equal(dbl.C, 2.0 * base.C)
    # identity: A = I (E4M3 1.0 on the diagonal, scale 2^0), K = N
    Kq = N = 64
    b2 = _rand_e4m3(rng, (N, Kq))
    sb2 = rng.integers(120, 135, (N, Kq // 32), dtype=np.uint8)
    eye = np.zeros((Kq, Kq), np.uint8)
    eye[np.arange(Kq), np.arange(Kq)] = 0x38
    res = orc.mxfp8(eye, np.full((Kq, Kq // 32), 127, np.uint8), b2, sb2)
    assert np.array_equal(res.C, _torch_dequant_e4m3(b2, sb2).T)
    # one-hot K: only k = 37 is non-zero in A, so C[m, n] = a[m,37] * b[n,37]
    a3 = np.zeros((M, K), np.uint8)
    a3[:, 37] = _rand_e4m3(rng, (M,))
    res3 = orc.mxfp8(a3, sa, b, sb)
    A3 = _torch_dequant_e4m3(a3, sa)
    B = _torch_dequant_e4m3(b, sb)
    assert np.array_equal(res3.C, np.outer(A3[:, 37], B[:, 37]))


def test_gemm_f16_matches_library_and_orientation(orc):
    """fp16 A [M,K] @ B [K,N]: equals numpy fp64 matmul; a transposed B would fail."""
    rng = np.random.default_rng(4)
    M, N, K = 24, 40, 72
    a = (rng.standard_normal((M, K))).astype(np.float16)
    b = (rng.standard_normal((K, N))).astype(np.float16)
    res = orc.gemm_f16(a, b)
    C = a.astype(np.float64) @ b.astype(np.float64)
    D = np.abs(a.astype(np.float64)) @ np.abs(b.astype(np.float64))
    assert res.C.shape == (M, N)
    assert np.all(np.abs(res.C - C) <= 1e-13 * D)
    assert np.array_equal(res.f16_bits, C.astype(np.float16).view(np.uint16)) or \
        np.mean(res.f16_bits == C.astype(np.float16).view(np.uint16)) > 0.99


def test_w4a16_matches_unpacked_values(orc):
    """Oracle on packed int4 equals fp64 matmul over the unpacked ints times 2^(s-127)."""
    M, N, K = 16, 48, 128
    d = synth.w4a16_inputs(M, N, K, seed=11)
    res = orc.w4a16(d["a"].numpy(), d["w"].numpy(), d["sw"].numpy())
    q = d["w_values"].numpy().astype(np.float64)
    s = 2.0 ** (d["sw"].numpy().astype(np.float64) - 127)
    W = q * np.repeat(s, 32, axis=1)
    A = d["a"].numpy().astype(np.float64)
    C = A @ W.T
    D = np.abs(A) @ np.abs(W).T
    assert np.all(np.abs(res.C - C) <= 1e-13 * D)


def test_w8_gemv_matches_library(orc):
    M, N, K = 5, 96, 256
    d = synth.w8_inputs(M, N, K, seed=12)
    res = orc.w8_gemv(d["x"].numpy(), d["w"].numpy(), d["sw"].numpy())
    q = d["w"].numpy().view(np.int8).astype(np.float64)
    s = 2.0 ** (d["sw"].numpy().astype(np.float64) - 127)
    W = q * np.repeat(s, 32, axis=1)
    X = d["x"].numpy().astype(np.float64)
    C = X @ W.T
    D = np.abs(X) @ np.abs(W).T
    assert np.all(np.abs(res.C - C) <= 1e-13 * D)
    assert np.allclose(res.D, D, rtol=1e-13)


# ---------------------------------------------------------------------------- tolerance
def test_tolerance_check_catches_planted_error(orc):
    """The element-wise check rejects a single wrong element and accepts fp16 rounding."""
    rng = np.random.default_rng(5)
    a = _rand_e4m3(rng, (16, 64))
    b = _rand_e4m3(rng, (32, 64))
    sa = np.full((16, 2), 124, np.uint8)
    sb = np.full((32, 2), 124, np.uint8)
    res = orc.mxfp8(a, sa, b, sb)
    ok, _, _ = orc.within_tolerance(res.f16.astype(np.float32), res)
    assert ok
    bad = res.f16.astype(np.float32).copy()
    bad[3, 7] += 0.01 * res.D[3, 7] + 1e-3
    ok, _, info = orc.within_tolerance(bad, res)
    assert not ok and info["n_bad"] == 1


def test_epilogue_hand_worked_example(orc):
    """Fused epilogue on a product worked out by hand: A = [[1, 2], [3, 4]] (E4M3 codes 0x38,
    0x40, 0x44, 0x48, scale 2^0, K padded to 32 with zeros), B = [[1, -1], [2, 0.5]].
    A B^T = [[1 - 2, 2 + 1], [3 - 4, 6 + 2]] = [[-1, 3], [-1, 8]]."""
    a = np.zeros((2, 32), np.uint8)
    a[0, :2] = [0x38, 0x40]          # 1, 2
    a[1, :2] = [0x44, 0x48]          # 3, 4
    b = np.zeros((2, 32), np.uint8)
    b[0, :2] = [0x38, 0xB8]          # 1, -1
    b[1, :2] = [0x40, 0x30]          # 2, 0.5
    s = np.full((2, 1), 127, np.uint8)
    res = orc.mxfp8(a, s, b, s)
    assert res.C.tolist() == [[-1.0, 3.0], [-1.0, 8.0]]
    # multiply_accumulate with C_old = [[0.5, -4], [1, -8]]: [[-0.5, -1], [0, 0]]
    old = np.array([[0.5, -4.0], [1.0, -8.0]], np.float16)
    acc = orc.epilogue(res, old)
    assert acc.C.tolist() == [[-0.5, -1.0], [0.0, 0.0]]
    assert acc.D.tolist() == [[3.5, 7.0], [8.0, 16.0]]    # sum |a b| (3, 3, 7, 8) + |C_old|
    # ReLU alone, then both
    assert orc.epilogue(res, relu=True).C.tolist() == [[0.0, 3.0], [0.0, 8.0]]
    both = orc.epilogue(res, old, relu=True)
    assert both.C.tolist() == [[0.0, 0.0], [0.0, 0.0]]
    assert not np.signbit(both.C).any()                    # ReLU of x <= 0 is +0
    assert both.f16_bits.tolist() == [[0, 0], [0, 0]]


def test_epilogue_invariants(orc):
    """Accumulating zeros is the plain product; accumulating -C (exact for integer products)
    then ReLU gives +0 everywhere; ReLU leaves positive entries unchanged."""
    g = np.random.default_rng(3)
    a = g.integers(-4, 5, (6, 64)).astype(np.float64)
    b = g.integers(-4, 5, (5, 64)).astype(np.float64)
    C, D = orc.dot_rows(a, b)
    res = orc.Result(C, D, None)
    z = orc.epilogue(res, np.zeros(C.shape, np.float16))
    assert np.array_equal(z.C, res.C) and np.array_equal(z.f16_bits, res.f16_bits)
    neg = orc.epilogue(res, (-C).astype(np.float16), relu=True)
    assert np.array_equal(neg.C, np.zeros_like(C))
    r = orc.epilogue(res, relu=True)
    assert np.array_equal(r.C[C > 0], C[C > 0]) and (r.C[C <= 0] == 0).all()


# OCP MX FP4 E2M1 by its definition: magnitudes of the 8 codes 0..7 (exponent field 0 is
# subnormal: 0, 0.5; then 1, 1.5, 2, 3, 4, 6), codes 8..15 the negatives.
E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e2m1_reference(code: int) -> float:
    v = E2M1_MAGNITUDES[code & 7]
    return -v if code & 8 else v


def test_e2m1_all_codes_match_definition(orc):
    t = orc.e2m1_table()
    for c in range(16):
        assert t[c] == _e2m1_reference(c) and np.signbit(t[c]) == bool(c & 8)


def test_e2m1_packing_even_k_in_low_nibble(orc):
    row = np.array([[0x71, 0xF8]], np.uint8)      # k0 = 0x1 (0.5), k1 = 0x7 (6), k2 = 0x8 (-0), k3 = 0xF (-6)
    d = orc.dequant(orc.E2M1, row, np.full((1, 1), 127, np.uint8), k=4)
    assert d.tolist() == [[0.5, 6.0, -0.0, -6.0]]
    d2 = orc.dequant(orc.E2M1, row, np.full((1, 1), 129, np.uint8), k=4)   # scale 2^2
    assert d2.tolist() == [[2.0, 24.0, -0.0, -24.0]]


def test_mxfp4_brute_force_exact_rationals(orc):
    rng = np.random.default_rng(7)
    for (M, N, K) in [(1, 1, 32), (3, 2, 64), (2, 4, 96)]:
        a = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
        b = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
        sa = rng.integers(115, 140, (M, K // 32), dtype=np.uint8)
        sb = rng.integers(115, 140, (N, K // 32), dtype=np.uint8)
        res = orc.mxfp4(a, sa, b, sb)

        def val(plane, scales, r, k):
            byte = int(plane[r, k // 2])
            code = byte & 15 if k % 2 == 0 else byte >> 4
            return Fraction(_e2m1_reference(code)) * Fraction(2) ** (int(scales[r, k // 32]) - 127)

        for m in range(M):
            for n in range(N):
                exact = sum(val(a, sa, m, k) * val(b, sb, n, k) for k in range(K))
                mag = sum(abs(val(a, sa, m, k) * val(b, sb, n, k)) for k in range(K))
                assert abs(Fraction(res.C[m, n]) - exact) <= Fraction(2.0 ** -50) * mag
                assert Fraction(res.D[m, n]) == pytest.approx(float(mag), rel=1e-14)


def test_mxfp4_matches_library_matmul(orc):
    """Decode with the literal table, multiply with numpy: the same product as the oracle."""
    rng = np.random.default_rng(8)
    M, N, K = 5, 7, 128
    a = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = rng.integers(120, 135, (M, K // 32), dtype=np.uint8)
    sb = rng.integers(120, 135, (N, K // 32), dtype=np.uint8)
    tab = np.array([_e2m1_reference(c) for c in range(16)])

    def decode(p, s):
        codes = np.stack([p & 15, p >> 4], axis=-1).reshape(p.shape[0], -1)
        return tab[codes] * np.exp2(np.repeat(s.astype(np.float64) - 127, 32, axis=1))

    want = decode(a, sa) @ decode(b, sb).T
    res = orc.mxfp4(a, sa, b, sb)
    assert np.allclose(res.C, want, rtol=1e-12, atol=1e-12)
    sel = orc.mxfp4(a, sa, b, sb, rows=np.array([4, 1]))
    assert np.array_equal(sel.C, res.C[[4, 1]])


# ------------------------------------------------- int4 with fp16 block scales (M2 recipe)
def _f16_rne(x: Fraction) -> Fraction:
    """Nearest binary16 value to an exact rational (ties to even), by Python's own half
    packing (struct 'e'), which is independent of the oracle's rounding routine."""
    import struct
    return Fraction(struct.unpack("<e", struct.pack("<e", float(x)))[0]) \
        if abs(x) < 65520 else None


def test_w4a16_f16s_hand_worked_fold(orc):
    """q = 7 with scale 1 + 2^-10: the exact product 7.0068359375 is not a half; the recipe's half
    multiply gives 7.0078125 (spacing 2^-8 between 4 and 8; 1793.75 rounds to 1794).  With every
    A element 1 over one block, C = 32 * 7.0078125 = 224.25 (the unrounded weights would give
    224.21875)."""
    w = np.full((1, 16), 0x77, np.uint8)
    s = np.array([[1 + 2.0 ** -10]], np.float16)
    assert np.all(orc.dequant_int4_f16s(w, s) == 7.0078125)
    a = np.ones((1, 32), np.float16)
    res = orc.w4a16_f16s(a, w, s)
    assert res.C[0, 0] == 224.25
    assert res.D[0, 0] == 224.25


def test_w4a16_f16s_power_of_two_scales_reduce_to_ue8m0(orc):
    """With every fp16 scale a power of two inside the exact range the product is the pinned
    UE8M0 W4A16 product, bit for bit."""
    M, N, K = 8, 40, 256
    d = synth.w4a16_inputs(M, N, K, seed=31)
    e = d["sw"].numpy().astype(np.int64)
    s16 = (2.0 ** (e - 127)).astype(np.float16)
    assert np.all(s16.astype(np.float64) == 2.0 ** (e - 127))
    a = d["a"].numpy()
    r1 = orc.w4a16_f16s(a, d["w"].numpy(), s16)
    r2 = orc.w4a16(a, d["w"].numpy(), d["sw"].numpy())
    assert np.array_equal(r1.C, r2.C) and np.array_equal(r1.D, r2.D)


def test_w4a16_f16s_brute_force_exact_rationals(orc):
    """Tiny random case: every weight rounded to half from the exact rational q * s, products
    summed exactly; the oracle's fp64 sum agrees to fp64 accuracy."""
    rng = np.random.default_rng(5)
    M, N, K = 3, 4, 64
    q = rng.integers(-8, 8, size=(N, K))
    s = (rng.standard_normal((N, K // 32)) * 0.37).astype(np.float16)
    s[0, 1] = np.float16(2.0 ** -14 * (1 + 2.0 ** -10))      # near the subnormal boundary
    s[1, 0] = np.float16(6.1e4)                               # q * s can overflow to inf
    q[1, :32] = np.clip(q[1, :32], -1, 1)                     # keep that block finite
    a = (rng.standard_normal((M, K))).astype(np.float16)
    packed = ((q[:, 0::2] & 0xF) | ((q[:, 1::2] & 0xF) << 4)).astype(np.uint8)
    res = orc.w4a16_f16s(a, packed, s)
    for m in range(M):
        for n in range(N):
            exact = Fraction(0)
            mag = Fraction(0)
            for k in range(K):
                wk = _f16_rne(Fraction(int(q[n, k])) * Fraction(float(s[n, k // 32])))
                p = Fraction(float(a[m, k])) * wk
                exact += p
                mag += abs(p)
            assert abs(Fraction(res.C[m, n]) - exact) <= Fraction(1, 2 ** 40) * (mag + 1)
            assert abs(Fraction(res.D[m, n]) - mag) <= Fraction(1, 2 ** 40) * (mag + 1)


def test_w4a16_f16s_matches_library_matmul(orc):
    """The oracle == numpy fp64 matmul over numpy's own half rounding of q * s, on the seeded
    workload recipe at a small size."""
    M, N, K = 16, 48, 256
    d = synth.w4a16_f16s_inputs(M, N, K, seed=13)
    q = d["w_values"].numpy().astype(np.float64)
    s = np.repeat(d["sw"].numpy().astype(np.float64), 32, axis=1)
    W = (q * s).astype(np.float16).astype(np.float64)
    A = d["a"].numpy().astype(np.float64)
    res = orc.w4a16_f16s(d["a"].numpy(), d["w"].numpy(), d["sw"].numpy())
    assert np.all(np.abs(res.C - A @ W.T) <= 1e-13 * (np.abs(A) @ np.abs(W).T))
    assert not np.all(np.abs(d["sw"].numpy().astype(np.float64)) ==
                      2.0 ** np.round(np.log2(np.abs(d["sw"].numpy().astype(np.float64)))))


# ----------------------------------------------------------------------- fused attention
def _attn_arrays(BH, Lq, Lk, d, seed, q_std=1.0):
    d_ = synth.attention_inputs(BH, Lq, Lk, d, seed, q_std=q_std)
    return d_["q"].numpy(), d_["k"].numpy(), d_["v"].numpy(), d_["scale"]


def test_attention_equal_keys_give_the_mean_of_v(orc):
    """All keys equal: every score of a row is the same, the softmax is uniform and O is the
    plain mean of the value rows."""
    q, k, v, scale = _attn_arrays(2, 5, 7, 16, seed=51)
    k[:] = k[:, :1, :]
    res = orc.attention(q, k, v, scale)
    want = np.repeat(v.astype(np.float64).mean(axis=1), 5, axis=0)
    assert np.allclose(res.C, want, rtol=0, atol=1e-14)


def test_attention_dominant_key_selects_its_value(orc):
    """One score 1000 above the rest: exp(-1000) underflows to 0 in fp64, so O is that key's
    value row exactly and D its magnitude."""
    d = 8
    q = np.zeros((1, 1, d), np.float16)
    q[0, 0, 0] = 1.0
    k = np.zeros((1, 4, d), np.float16)
    k[0, 2, 0] = 1000.0
    v = np.arange(32, dtype=np.float16).reshape(1, 4, d) - 10
    res = orc.attention(q, k, v, 1.0)
    assert np.array_equal(res.C[0], v[0, 2].astype(np.float64))
    assert np.array_equal(res.D[0], np.abs(v[0, 2].astype(np.float64)))


def test_attention_matches_library_sdpa(orc):
    """torch's scaled_dot_product_attention in fp64 (a library routine) on decoded fp16 data."""
    q, k, v, scale = _attn_arrays(3, 37, 53, 32, seed=52, q_std=3.0)
    res = orc.attention(q, k, v, scale)
    t = [torch.from_numpy(x.astype(np.float64)) for x in (q, k, v)]
    ref = torch.nn.functional.scaled_dot_product_attention(t[0], t[1], t[2], scale=scale)
    assert np.allclose(res.C, ref.reshape(-1, 32).numpy(), rtol=0, atol=1e-12)


def test_attention_invariants(orc):
    """Permuting keys together with their values leaves O unchanged; a per-row shift of every
    score (a key component shared by all keys) leaves O unchanged."""
    q, k, v, scale = _attn_arrays(1, 6, 40, 16, seed=53, q_std=2.0)
    base = orc.attention(q, k, v, scale).C
    perm = np.random.default_rng(0).permutation(40)
    assert np.allclose(orc.attention(q, k[:, perm], v[:, perm], scale).C, base, atol=1e-13)
    k2 = k.copy()
    k2[:, :, 15] = 1.0
    q0 = q.copy()
    q0[:, :, 15] = 0.0
    q1 = q.copy()
    q1[:, :, 15] = np.linspace(-4, 4, 6).astype(np.float16)
    assert np.allclose(orc.attention(q0, k2, v, scale).C, orc.attention(q1, k2, v, scale).C,
                       atol=1e-13)


def test_attention_high_precision_tiny(orc):
    """A tiny case against 50-digit arithmetic (mpmath) of the same definition."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    q, k, v, scale = _attn_arrays(1, 3, 5, 4, seed=54, q_std=2.0)
    res = orc.attention(q, k, v, scale)
    for i in range(3):
        s = [mpmath.mpf(scale) * sum(mpmath.mpf(float(q[0, i, c])) * mpmath.mpf(float(k[0, j, c]))
                                     for c in range(4)) for j in range(5)]
        m = max(s)
        p = [mpmath.e ** (x - m) for x in s]
        l = sum(p)
        for c in range(4):
            o = sum(p[j] * mpmath.mpf(float(v[0, j, c])) for j in range(5)) / l
            assert abs(float(o) - res.C[i, c]) <= 1e-14
