"""GPU parity: every kernel of the library against the CPU oracle, through the C ABI.

Tolerance (element-wise): |C_gpu - C| <= 2e-3 * sum_k |a_mk b_nk| + 2^-24, with C the fp64
product of the decoded operands; non-finite values must match.  Decoded operands must match bit
for bit (dequantise-only debug kernel).
"""
import numpy as np
import pytest
import torch

import block_scaled_quantized_tcgen05_gb300 as q
from block_scaled_quantized_tcgen05_gb300 import synth

pytestmark = pytest.mark.gpu

REL = 2e-3


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from block_scaled_quantized_tcgen05_gb300 import build
    build.build()
    q.load_library()
    q.qgemm_set_wait_timeout_ns(2_000_000_000)
    return torch.device("cuda:0")


def _check(got: torch.Tensor, res, orc, rows=None, what=""):
    code = q.qgemm_poll_device_error()
    assert code == 0, f"{what}: a device wait timed out (error word {code:#x})"
    ok, worst, info = orc.within_tolerance(got.float().cpu().numpy(), res, REL, rows)
    assert ok, f"{what}: {info}"
    return worst


def _mx_views(d, dev):
    a, sa, b, sb = (d[k].to(dev) for k in ("a", "sa", "b", "sb"))
    return q.qgemm_create_tensor(q.E4M3, a, sa), q.qgemm_create_tensor(q.E4M3, b, sb), (a, sa, b, sb)


# ----------------------------------------------------------------------- dequant debug
def test_dequant_debug_bit_exact_all_codes(dev, orc):
    rows, K = 256, 256
    data = torch.arange(rows * K, dtype=torch.int64).remainder(256).to(torch.uint8).reshape(rows, K)
    data = data[torch.randperm(rows, generator=synth.generator(1))].contiguous()
    sc = torch.randint(0, 247, (rows, K // 32), generator=synth.generator(2), dtype=torch.uint8)
    sc[0, 0] = 255                                               # NaN scale
    for dt in (q.E4M3, q.INT8):
        t = q.qgemm_create_tensor(dt, data.to(dev), sc.to(dev))
        out = torch.empty(rows, K, dtype=torch.float32, device=dev)
        q.qgemm_dequant_debug(t, out)
        ref = orc.dequant(orc.E4M3 if dt == q.E4M3 else orc.INT8, data.numpy(), sc.numpy())
        got = out.cpu().numpy().astype(np.float64)
        assert np.array_equal(np.isnan(got), np.isnan(ref))
        fin = ~np.isnan(ref)
        assert np.array_equal(got[fin], ref[fin].astype(np.float32).astype(np.float64))
    # int4: every nibble value in both positions
    sc4 = torch.randint(100, 150, (rows, 2 * K // 32), generator=synth.generator(3),
                        dtype=torch.uint8)
    t4 = q.qgemm_create_tensor(q.INT4, data.to(dev), sc4.to(dev))
    out4 = torch.empty(rows, 2 * K, dtype=torch.float32, device=dev)
    q.qgemm_dequant_debug(t4, out4)
    ref4 = orc.dequant(orc.INT4, data.numpy(), sc4.numpy())
    assert np.array_equal(out4.cpu().numpy().astype(np.float64), ref4)
    # fp16 view: the values themselves
    h = torch.randn(64, 96, generator=synth.generator(4)).half()
    th = q.qgemm_create_tensor(q.F16, h.to(dev), None)
    outh = torch.empty(64, 96, dtype=torch.float32, device=dev)
    q.qgemm_dequant_debug(th, outh)
    assert torch.equal(outh.cpu(), h.float())


# ------------------------------------------------------------------------------ MXFP8
@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (300, 520, 416), (128, 96, 64),
                                   (1, 1, 32), (257, 384, 1024), (640, 768, 256)])
def test_mxfp8_matches_oracle(dev, orc, M, N, K):
    d = synth.mxfp8_inputs(M, N, K, seed=M + N + K, row_variance=True)
    A, B, _ = _mx_views(d, dev)
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
    q.qgemm_mxfp8(A, B, C)
    res = orc.mxfp8(d["a"].numpy(), d["sa"].numpy(), d["b"].numpy(), d["sb"].numpy())
    _check(C, res, orc, what=f"mxfp8 {M}x{N}x{K}")
    assert orc.cosine(C.float().cpu().numpy(), res.C) > 0.99999


def test_mxfp8_padded_strides_and_output(dev, orc):
    M, N, K = 200, 264, 256
    d = synth.mxfp8_inputs(M, N, K, seed=5)
    a = torch.zeros(M, K + 64, dtype=torch.uint8)
    a[:, :K] = d["a"]
    sa = torch.full((M, 16), 127, dtype=torch.uint8)
    sa[:, :K // 32] = d["sa"]
    A = q.qgemm_create_tensor(q.E4M3, a.to(dev)[:, :K], sa.to(dev)[:, :K // 32])
    B = q.qgemm_create_tensor(q.E4M3, d["b"].to(dev), d["sb"].to(dev))
    Cbig = torch.full((M, N + 40), 7.0, dtype=torch.float16, device=dev)
    q.qgemm_mxfp8(A, B, Cbig[:, :N])
    res = orc.mxfp8(d["a"].numpy(), d["sa"].numpy(), d["b"].numpy(), d["sb"].numpy())
    _check(Cbig[:, :N], res, orc, what="mxfp8 strided")
    assert torch.all(Cbig[:, N:] == 7.0)                        # nothing written past N


def test_mxfp8_invariants(dev, orc):
    M, N, K = 256, 512, 512
    d = synth.mxfp8_inputs(M, N, K, seed=21)
    A, B, (a, sa, b, sb) = _mx_views(d, dev)
    C = torch.empty(M, N, dtype=torch.float16, device=dev)
    q.qgemm_mxfp8(A, B, C)
    # doubling every A scale doubles C exactly (away from the fp16 subnormal range)
    A2 = q.qgemm_create_tensor(q.E4M3, a, sa + 1)
    C2 = torch.empty_like(C)
    q.qgemm_mxfp8(A2, B, C2)
    big = C.abs() >= 2.0 ** -13
    assert torch.equal(C2[big], 2 * C[big])
    # identity A (E4M3 1.0, scale 2^0), K = N: C = fp16(deq(B)^T)
    Ki = 256
    bi = d["b"][:, :Ki].contiguous()
    sbi = d["sb"][:, :Ki // 32].contiguous()
    eye = torch.zeros(Ki, Ki, dtype=torch.uint8)
    eye[torch.arange(Ki), torch.arange(Ki)] = 0x38
    Ai = q.qgemm_create_tensor(q.E4M3, eye.to(dev), torch.full((Ki, Ki // 32), 127, dtype=torch.uint8, device=dev))
    Bi = q.qgemm_create_tensor(q.E4M3, bi.to(dev), sbi.to(dev))
    Ci = torch.empty(Ki, N, dtype=torch.float16, device=dev)
    q.qgemm_mxfp8(Ai, Bi, Ci)
    want = orc.f16_rn(orc.dequant(orc.E4M3, bi.numpy(), sbi.numpy()).T.copy())
    assert np.array_equal(Ci.cpu().numpy().view(np.uint16), want)
    # one-hot K: C = fp16(a[:, 37] * b[:, 37])
    a1 = torch.zeros_like(d["a"])
    a1[:, 37] = d["a"][:, 37]
    A1 = q.qgemm_create_tensor(q.E4M3, a1.to(dev), sa)
    C1 = torch.empty_like(C)
    q.qgemm_mxfp8(A1, B, C1)
    res1 = orc.mxfp8(a1.numpy(), d["sa"].numpy(), d["b"].numpy(), d["sb"].numpy())
    assert np.array_equal(C1.cpu().numpy().view(np.uint16), res1.f16_bits)
    # slicing rows of A and B (data and scales together) gives exactly the matching block of C
    As = q.qgemm_tensor_slice(A, 64, 100, 0, K)
    Bs = q.qgemm_tensor_slice(B, 128, 200, 0, K)
    Cs = torch.empty(100, 200, dtype=torch.float16, device=dev)
    q.qgemm_mxfp8(As, Bs, Cs)
    assert torch.equal(Cs, C[64:164, 128:328])
    # slicing K into halves: C ~ C_lo + C_hi
    Alo, Ahi = q.qgemm_tensor_slice(A, 0, M, 0, K // 2), q.qgemm_tensor_slice(A, 0, M, K // 2, K // 2)
    Blo, Bhi = q.qgemm_tensor_slice(B, 0, N, 0, K // 2), q.qgemm_tensor_slice(B, 0, N, K // 2, K // 2)
    Clo, Chi = torch.empty_like(C), torch.empty_like(C)
    q.qgemm_mxfp8(Alo, Blo, Clo)
    q.qgemm_mxfp8(Ahi, Bhi, Chi)
    res = orc.mxfp8(d["a"].numpy(), d["sa"].numpy(), d["b"].numpy(), d["sb"].numpy())
    ok, _, info = orc.within_tolerance((Clo.float() + Chi.float()).cpu().numpy(), res, 2 * REL)
    assert ok, info


def test_mxfp8_edge_cases(dev, orc):
    d = synth.mxfp8_inputs(64, 128, 64, seed=9)
    A, B, _ = _mx_views(d, dev)
    # K = 0: the empty sum is zero
    A0 = q.qgemm_create_tensor(q.E4M3, torch.zeros(64, 16, dtype=torch.uint8, device=dev),
                               torch.zeros(64, 4, dtype=torch.uint8, device=dev), k=0)
    B0 = q.qgemm_create_tensor(q.E4M3, torch.zeros(128, 16, dtype=torch.uint8, device=dev),
                               torch.zeros(128, 4, dtype=torch.uint8, device=dev), k=0)
    C = torch.full((64, 128), 3.0, dtype=torch.float16, device=dev)
    q.qgemm_mxfp8(A0, B0, C)
    torch.cuda.synchronize()
    assert torch.all(C == 0)
    # M = 0: nothing happens
    Ae = q.qgemm_tensor_slice(A, 0, 0, 0, 64)
    q.qgemm_mxfp8(Ae, B, C[:0])
    # NaN propagation: an E4M3 NaN code or a 0xFF scale poisons its row
    a = d["a"].clone()
    sa = d["sa"].clone()
    a[3, 5] = 0x7F
    sa[7, 1] = 255
    An = q.qgemm_create_tensor(q.E4M3, a.to(dev), sa.to(dev))
    Cn = torch.empty(64, 128, dtype=torch.float16, device=dev)
    q.qgemm_mxfp8(An, B, Cn)
    Cn = Cn.cpu()
    assert torch.isnan(Cn[3]).all() and torch.isnan(Cn[7]).all()
    assert not torch.isnan(Cn[[0, 1, 2, 4, 5, 6]]).any()
    # wrong argument: error status, no launch
    with pytest.raises(q.QGemmError) as ei:
        q.qgemm_mxfp8(A, q.qgemm_tensor_slice(B, 0, 128, 0, 32), C)
    assert ei.value.name == "QGEMM_ERR_INVALID_ARG"


def test_mxfp8_many_tiles_offset_k(dev, orc):
    """More output tiles than CTA pairs, a K window starting one scale byte into the planes and a
    ragged last k-tile; two calls in a row give identical bits."""
    M, N, K0, K = 2344, 2552, 32, 1056
    d = synth.mxfp8_inputs(M, N, K0 + K, seed=77, row_variance=True)
    A, B, _ = _mx_views(d, dev)
    As = q.qgemm_tensor_slice(A, 0, M, K0, K)
    Bs = q.qgemm_tensor_slice(B, 0, N, K0, K)
    C = torch.empty(M, N, dtype=torch.float16, device=dev)
    q.qgemm_mxfp8(As, Bs, C)
    C2 = torch.empty_like(C)
    q.qgemm_mxfp8(As, Bs, C2)
    assert torch.equal(C, C2)
    rows = np.array([0, 1, 127, 128, 255, 256, 1000, 2047, 2048, 2303, 2304, 2343])
    a = d["a"][:, K0:].contiguous()
    sa = d["sa"][:, K0 // 32:].contiguous()
    b = d["b"][:, K0:].contiguous()
    sb = d["sb"][:, K0 // 32:].contiguous()
    res = orc.mxfp8(a.numpy(), sa.numpy(), b.numpy(), sb.numpy(), rows=rows)
    _check(C[torch.from_numpy(rows).to(dev)], res, orc, what="mxfp8 many tiles, K offset")


def test_mxfp8_full_size_sampled(dev, orc):
    """8192^3 with per-row variance 10^U(-2,2): full GPU product, oracle on sampled rows."""
    d = synth.workload("mxfp8_8192")
    A, B, _ = _mx_views(d, dev)
    C = torch.empty(8192, 8192, dtype=torch.float16, device=dev)
    q.qgemm_mxfp8(A, B, C)
    rows = np.sort(np.random.default_rng(0).choice(8192, 48, replace=False))
    rows = np.concatenate([[0, 127, 128, 8191], rows])
    res = orc.mxfp8(d["a"].numpy(), d["sa"].numpy(), d["b"].numpy(), d["sb"].numpy(), rows=rows)
    got = C[torch.from_numpy(rows).to(dev)]
    _check(got, res, orc, what="mxfp8 8192^3 sampled")
    # the whole product is repeatable bit for bit (no timing-dependent stage reuse)
    for _ in range(2):
        C2 = torch.empty_like(C)
        q.qgemm_mxfp8(A, B, C2)
        assert torch.equal(C2.view(torch.int16), C.view(torch.int16))


@pytest.mark.parametrize("epi", [None, (True, True)])
def test_mxfp8_last_wave_half_tiles(dev, orc, epi):
    """2048 x 3072 has 96 pair tiles: 76 whole ones, then 20 left over, each run as two 256 x 128
    halves.  Every element against the oracle, and the columns of the split tiles bit-identical
    to the same columns computed as whole tiles (B sliced to its last 768 rows: 24 whole tiles)."""
    M, N, K = 2048, 3072, 256
    d = synth.mxfp8_inputs(M, N, K, seed=61, row_variance=True)
    A, B, (a, sa, b, sb) = _mx_views(d, dev)
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
    c_old = (torch.randn(M, N, generator=synth.generator(62)) * 3).to(torch.float16)
    if epi:
        C.copy_(c_old.to(dev))
        q.qgemm_mxfp8_ex(A, B, C, accumulate=True, relu=True)
    else:
        q.qgemm_mxfp8(A, B, C)
    res = orc.mxfp8(d["a"].numpy(), d["sa"].numpy(), d["b"].numpy(), d["sb"].numpy())
    if epi:
        res = orc.epilogue(res, c_old.numpy(), relu=True)
    _check(C, res, orc, what=f"mxfp8 half tiles epi={epi}")
    Bs = q.qgemm_tensor_slice(B, 2304, 768, 0, K)
    Cs = torch.full((M, 768), float("nan"), dtype=torch.float16, device=dev)
    if epi:
        Cs.copy_(c_old[:, 2304:].to(dev))
        q.qgemm_mxfp8_ex(A, Bs, Cs, accumulate=True, relu=True)
    else:
        q.qgemm_mxfp8(A, Bs, Cs)
    torch.cuda.synchronize()
    assert torch.equal(Cs.view(torch.int16), C[:, 2304:].view(torch.int16))


# ------------------------------------------------------------------------------- fp16
# (1024, 4864, 128): exactly one wave of 256 x 256 pair tiles on 76 pairs
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 328, 200), (96, 64, 512),
                                   (384, 512, 1024), (1024, 4864, 128)])
def test_gemm_f16_matches_oracle(dev, orc, M, N, K):
    d = synth.f16_inputs(M, N, K, seed=M * 7 + N)
    C = torch.empty(M, N, dtype=torch.float16, device=dev)
    q.gemm_f16(d["a"].to(dev), d["b"].to(dev), C)
    res = orc.gemm_f16(d["a"].numpy(), d["b"].numpy())
    _check(C, res, orc, what=f"f16 {M}x{N}x{K}")


def test_gemm_f16_full_size_sampled(dev, orc):
    d = synth.workload("f16_4096")
    C = torch.empty(4096, 4096, dtype=torch.float16, device=dev)
    q.gemm_f16(d["a"].to(dev), d["b"].to(dev), C)
    rows = np.concatenate([[0, 4095], np.sort(np.random.default_rng(1).choice(4096, 30, replace=False))])
    res = orc.gemm_f16(d["a"].numpy(), d["b"].numpy(), rows=rows)
    _check(C[torch.from_numpy(rows).to(dev)], res, orc, what="f16 4096^3 sampled")
    C2 = torch.empty_like(C)
    q.gemm_f16(d["a"].to(dev), d["b"].to(dev), C2)
    assert torch.equal(C2.view(torch.int16), C.view(torch.int16))     # repeatable bit for bit


@pytest.mark.parametrize("M,N,K", [(2560, 2048, 512), (2304, 2144, 320)])
def test_gemm_f16_last_wave_halves(dev, orc, M, N, K):
    """More pair tiles than one wave (80 and 81 tiles on 76 pairs): the leftover tiles run as two
    256 x 128 halves each (for N = 2144 one half lies wholly past N); every output checked."""
    d = synth.f16_inputs(M, N, K, seed=M + N)
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
    q.gemm_f16(d["a"].to(dev), d["b"].to(dev), C)
    res = orc.gemm_f16(d["a"].numpy(), d["b"].numpy())
    _check(C, res, orc, what=f"f16 {M}x{N}x{K} last-wave halves")
    C2 = torch.empty_like(C)
    q.gemm_f16(d["a"].to(dev), d["b"].to(dev), C2)
    assert torch.equal(C2.view(torch.int16), C.view(torch.int16))


# ------------------------------------------------------------------------------ W4A16
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 300, 256), (256, 640, 1024)])
def test_w4a16_matches_oracle(dev, orc, M, N, K):
    d = synth.w4a16_inputs(M, N, K, seed=M + 3 * N)
    W = q.qgemm_create_tensor(q.INT4, d["w"].to(dev), d["sw"].to(dev))
    C = torch.empty(M, N, dtype=torch.float16, device=dev)
    q.qgemm_w4a16(d["a"].to(dev), W, C)
    res = orc.w4a16(d["a"].numpy(), d["w"].numpy(), d["sw"].numpy())
    _check(C, res, orc, what=f"w4a16 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(300, 640, 1536), (1000, 1000, 512), (129, 136, 512)])
def test_w4a16_pair_path_ragged(dev, orc, M, N, K):
    """Shapes of the CTA-pair route (N > 128, K % 512 == 0, aligned scale rows) with
    ragged token and weight tiles and several scale groups."""
    d = synth.w4a16_inputs(M, N, K, seed=7 * M + N)
    W = q.qgemm_create_tensor(q.INT4, d["w"].to(dev), d["sw"].to(dev))
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
    q.qgemm_w4a16(d["a"].to(dev), W, C)
    res = orc.w4a16(d["a"].numpy(), d["w"].numpy(), d["sw"].numpy())
    _check(C, res, orc, what=f"w4a16 pair {M}x{N}x{K}")


@pytest.mark.parametrize("scale_pad", [0, 9])
def test_w4a16_one_cta_route_several_tiles_per_cta(dev, orc, scale_pad):
    """K % 512 != 0 takes the one-CTA route with cp.async staging; 16 x 10 = 160 tiles of
    128 x 256 on at most 152 CTAs, so some CTAs walk two tiles and the tile and k counters roll
    over.  scale_pad = 9: scale rows 9 bytes apart (not 4-byte aligned), the byte-load instance."""
    M, N, K = 2048, 2560, 256
    nblk = K // 32
    d = synth.w4a16_inputs(M, N, K, seed=1234 + scale_pad)
    if scale_pad:
        s_full = torch.full((N, scale_pad), 255, dtype=torch.uint8)
        s_full[:, :nblk] = d["sw"]
        sv = s_full.to(dev)[:, :nblk]
    else:
        sv = d["sw"].to(dev)
    W = q.qgemm_create_tensor(q.INT4, d["w"].to(dev), sv)
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
    q.qgemm_w4a16(d["a"].to(dev), W, C)
    rows = np.concatenate([np.arange(0, 8), np.arange(M - 8, M),
                           np.sort(np.random.default_rng(3).choice(M, 48, replace=False))])
    res = orc.w4a16(d["a"].numpy()[rows], d["w"].numpy(), d["sw"].numpy())
    _check(C[torch.from_numpy(rows).to(dev)], res, orc, what=f"w4a16 one-CTA route lds pad {scale_pad}")
    assert not torch.isnan(C).any()


def test_w4a16_scales_outside_fused_window(dev, orc):
    """Scale exponents on both sides of the fused conversion's window (117..132) take the exact
    general path; every block gets one of 104, 110, 116, 117, 132, 133, 139."""
    M, N, K = 256, 384, 1024
    d = synth.w4a16_inputs(M, N, K, seed=99)
    exps = torch.tensor([104, 110, 116, 117, 132, 133, 139], dtype=torch.uint8)
    sw = exps[torch.randint(0, 7, d["sw"].shape, generator=synth.generator(5))].contiguous()
    a = (d["a"].float() * 2.0 ** -6).to(torch.float16)      # keep products inside fp16 range
    W = q.qgemm_create_tensor(q.INT4, d["w"].to(dev), sw.to(dev))
    C = torch.empty(M, N, dtype=torch.float16, device=dev)
    q.qgemm_w4a16(a.to(dev), W, C)
    res = orc.w4a16(a.numpy(), d["w"].numpy(), sw.numpy())
    _check(C, res, orc, what="w4a16 extreme scales")


def test_w4a16_full_size_sampled(dev, orc):
    d = synth.workload("w4a16_prefill")
    W = q.qgemm_create_tensor(q.INT4, d["w"].to(dev), d["sw"].to(dev))
    C = torch.empty(4096, 14336, dtype=torch.float16, device=dev)
    q.qgemm_w4a16(d["a"].to(dev), W, C)
    rows = np.concatenate([[0, 4095], np.sort(np.random.default_rng(2).choice(4096, 14, replace=False))])
    res = orc.w4a16(d["a"].numpy(), d["w"].numpy(), d["sw"].numpy(), rows=rows)
    _check(C[torch.from_numpy(rows).to(dev)], res, orc, what="w4a16 sampled")
    for _ in range(2):                                                  # repeatable bit for bit
        C2 = torch.empty_like(C)
        q.qgemm_w4a16(d["a"].to(dev), W, C2)
        assert torch.equal(C2.view(torch.int16), C.view(torch.int16))


# ------------------------------------------------------------------------------- GEMV
@pytest.mark.parametrize("M", [1, 3, 8, 9, 16])
def test_w8_gemv_matches_oracle(dev, orc, M):
    N, K = 1000, 1056
    d = synth.w8_inputs(M, N, K, seed=M)
    W = q.qgemm_create_tensor(q.INT8, d["w"].to(dev), d["sw"].to(dev))
    Y = torch.empty(M, N, dtype=torch.float16, device=dev)
    q.qgemm_w8_gemv(d["x"].to(dev), W, Y)
    res = orc.w8_gemv(d["x"].numpy(), d["w"].numpy(), d["sw"].numpy())
    _check(Y, res, orc, what=f"w8 gemv M={M}")


def test_w8_gemv_extreme_scales(dev, orc):
    """Per-block fp32 scaling handles every scale byte exactly (no fp16 folding)."""
    M, N, K = 4, 64, 256
    d = synth.w8_inputs(M, N, K, seed=99)
    sw = torch.randint(60, 200, d["sw"].shape, generator=synth.generator(5), dtype=torch.uint8)
    sw[3, 2] = 255          # NaN scale: row 3 of W poisons column 3 of Y
    sw[5, 0] = 0            # subnormal 2^-127 scale
    sw[9, 7] = 254
    W = q.qgemm_create_tensor(q.INT8, d["w"].to(dev), sw.to(dev))
    Y = torch.empty(M, N, dtype=torch.float16, device=dev)
    q.qgemm_w8_gemv(d["x"].to(dev), W, Y)
    res = orc.w8_gemv(d["x"].numpy(), d["w"].numpy(), sw.numpy())
    _check(Y, res, orc, what="w8 gemv extreme scales")
    assert torch.isnan(Y[:, 3].cpu()).all() and not torch.isnan(Y[:, 4].cpu()).any()


@pytest.mark.parametrize("M,scale_pad", [(2, 48), (16, 48), (5, 36), (12, 40)])
def test_w8_gemv_padded_strides_and_repeatable(dev, orc, M, scale_pad):
    """Views into wider buffers: weight rows K + 64 bytes apart, X rows K + 24 halves apart and
    scale rows `scale_pad` bytes apart (48: 16-byte aligned rows whose 33 blocks end inside a
    16-byte group; 36: 4-byte aligned; 40: 8-byte aligned).  N = 200 leaves a partial 64-row
    block.  Two calls give bit-identical outputs."""
    N, K = 200, 1056
    nblk = K // 32
    d = synth.w8_inputs(M, N, K, seed=40 + M)
    w_full = torch.zeros(N, K + 64, dtype=torch.uint8)
    w_full[:, :K] = d["w"]
    s_full = torch.full((N, scale_pad), 255, dtype=torch.uint8)     # padding would poison as NaN
    s_full[:, :nblk] = d["sw"]
    x_full = torch.zeros(M, K + 24, dtype=torch.float16)
    x_full[:, :K] = d["x"]
    wv, sv, xv = w_full.to(dev)[:, :K], s_full.to(dev)[:, :nblk], x_full.to(dev)[:, :K]
    W = q.qgemm_create_tensor(q.INT8, wv, sv)
    Y = torch.empty(M, N, dtype=torch.float16, device=dev)
    q.qgemm_w8_gemv(xv, W, Y)
    res = orc.w8_gemv(d["x"].numpy(), d["w"].numpy(), d["sw"].numpy())
    _check(Y, res, orc, what=f"w8 gemv padded M={M} lds={scale_pad}")
    Y2 = torch.empty_like(Y)
    q.qgemm_w8_gemv(xv, W, Y2)
    assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16))


@pytest.mark.parametrize("M", [1, 8, 16])
def test_w8_gemv_full_size_sampled(dev, orc, M):
    d = synth.workload("w8_decode", M=M)
    W = q.qgemm_create_tensor(q.INT8, d["w"].to(dev), d["sw"].to(dev))
    Y = torch.empty(M, 28672, dtype=torch.float16, device=dev)
    q.qgemm_w8_gemv(d["x"].to(dev), W, Y)
    cols = np.concatenate([[0, 28671], np.sort(np.random.default_rng(M).choice(28672, 2046, replace=False))])
    res = orc.w8_gemv(d["x"].numpy(), d["w"].numpy()[cols], d["sw"].numpy()[cols])
    _check(Y[:, torch.from_numpy(cols).to(dev)], res, orc, what=f"w8 gemv 28672x8192 M={M}")
    # every output is repeatable bit for bit: a stage handed back to the producer before its reads
    # are ordered shows up here as whole 64-row blocks that change from call to call
    for _ in range(8):
        Y2 = torch.empty_like(Y)
        q.qgemm_w8_gemv(d["x"].to(dev), W, Y2)
        assert torch.equal(Y2.view(torch.int16), Y.view(torch.int16))


# -------------------------------------------------------------------- failure detection
def test_bounded_wait_gives_up_and_context_survives(dev, orc):
    q.qgemm_poll_device_error()
    q.qgemm_selftest_wait_timeout(2_000_000)            # 2 ms on a barrier nothing completes
    code = q.qgemm_poll_device_error()
    assert code & 16
    assert q.qgemm_poll_device_error() == 0             # cleared
    d = synth.mxfp8_inputs(128, 256, 128, seed=0)
    A, B, _ = _mx_views(d, dev)
    C = torch.empty(128, 256, dtype=torch.float16, device=dev)
    q.qgemm_mxfp8(A, B, C)
    res = orc.mxfp8(d["a"].numpy(), d["sa"].numpy(), d["b"].numpy(), d["sb"].numpy())
    _check(C, res, orc, what="after self-test")


def test_sm_clock_probe_reads_a_plausible_clock(dev):
    """The clock probe's cycles over its window give an SM clock between 0.3 and 2.6 GHz (the
    GPU's maximum is 2.07 GHz), and the window it measured is at least the one asked for."""
    out = torch.zeros(2, dtype=torch.int64, device=dev)
    q.qgemm_sm_clock_probe(200_000, out)
    torch.cuda.synchronize()
    cycles, ns = (int(v) for v in out.cpu())
    assert ns >= 200_000
    assert 0.3 < cycles / ns < 2.6, (cycles, ns)
