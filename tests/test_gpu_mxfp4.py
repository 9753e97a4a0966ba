"""GPU parity of the MXFP4 GEMM (E2M1 data packed two per byte, UE8M0 scale per 32 along K)
against the CPU oracle, through the C ABI.

Tolerance (element-wise): |C_gpu - C| <= 2e-3 * sum_k |a_mk b_nk| + 2^-24, C the fp64 product of
the decoded operands; non-finite values must match.  The decoded operands must match the oracle's
E2M1 decoding bit for bit (dequantise-only debug kernel, which uses the hardware conversion).
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


def _check(got, res, orc, rows=None, what=""):
    code = q.qgemm_poll_device_error()
    assert code == 0, f"{what}: a device wait timed out (error word {code:#x})"
    ok, worst, info = orc.within_tolerance(got.float().cpu().numpy(), res, REL, rows)
    assert ok, f"{what}: {info}"
    return worst


def _views(d, dev):
    a, sa, b, sb = (d[k].to(dev) for k in ("a", "sa", "b", "sb"))
    return q.qgemm_create_tensor(q.E2M1, a, sa), q.qgemm_create_tensor(q.E2M1, b, sb), (a, sa, b, sb)


def _oracle(orc, d, rows=None):
    return orc.mxfp4(d["a"].numpy(), d["sa"].numpy(), d["b"].numpy(), d["sb"].numpy(), rows=rows)


def test_dequant_debug_e2m1_bit_exact(dev, orc):
    """Every byte value (so every code in both nibble positions) under random scales, NaN scale
    byte included."""
    rows, KB = 256, 128
    data = torch.arange(rows * KB, dtype=torch.int64).remainder(256).to(torch.uint8)
    data = data.reshape(rows, KB)[torch.randperm(rows, generator=synth.generator(31))].contiguous()
    sc = torch.randint(60, 200, (rows, 2 * KB // 32), generator=synth.generator(32),
                       dtype=torch.uint8)
    sc[5, 3] = 255
    t = q.qgemm_create_tensor(q.E2M1, data.to(dev), sc.to(dev))
    out = torch.empty(rows, 2 * KB, dtype=torch.float32, device=dev)
    q.qgemm_dequant_debug(t, out)
    ref = orc.dequant(orc.E2M1, data.numpy(), sc.numpy())
    got = out.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin].astype(np.float32).astype(np.float64))


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (300, 520, 416), (128, 96, 64), (1, 1, 32),
                                   (96, 200, 256), (257, 384, 1024), (640, 768, 544)])
def test_mxfp4_matches_oracle(dev, orc, M, N, K):
    d = synth.mxfp4_inputs(M, N, K, seed=M + 3 * N + K, row_variance=True)
    A, B, _ = _views(d, dev)
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
    q.qgemm_mxfp4(A, B, C)
    res = _oracle(orc, d)
    _check(C, res, orc, what=f"mxfp4 {M}x{N}x{K}")
    assert orc.cosine(C.float().cpu().numpy(), res.C) > 0.99999


def test_mxfp4_many_tiles_offset_k_strided(dev, orc):
    """More output tiles than CTA pairs; a K window starting one scale block into the planes
    (16 bytes into each packed row) with a ragged last stage; a padded output row stride; two
    calls give identical bits."""
    M, N, K0, K = 2344, 2552, 32, 1056
    d = synth.mxfp4_inputs(M, N, K0 + K, seed=78, row_variance=True)
    A, B, _ = _views(d, dev)
    As = q.qgemm_tensor_slice(A, 0, M, K0, K)
    Bs = q.qgemm_tensor_slice(B, 0, N, K0, K)
    Cbig = torch.full((M, N + 24), 5.0, dtype=torch.float16, device=dev)
    C = Cbig[:, :N]
    q.qgemm_mxfp4(As, Bs, C)
    C2 = torch.empty(M, N, dtype=torch.float16, device=dev)
    q.qgemm_mxfp4(As, Bs, C2)
    assert torch.equal(C, C2)
    assert torch.all(Cbig[:, N:] == 5.0)
    rows = np.array([0, 1, 127, 128, 255, 256, 1000, 2047, 2048, 2303, 2304, 2343])
    sub = {"a": d["a"][:, K0 // 2:].contiguous(), "sa": d["sa"][:, K0 // 32:].contiguous(),
           "b": d["b"][:, K0 // 2:].contiguous(), "sb": d["sb"][:, K0 // 32:].contiguous()}
    res = _oracle(orc, sub, rows)
    _check(C[torch.from_numpy(rows).to(dev)], res, orc, what="mxfp4 many tiles, K offset")


def test_mxfp4_scale_invariant(dev, orc):
    """Raising every A scale byte by one doubles C exactly (fp16 normal range)."""
    M, N, K = 256, 512, 512
    d = synth.mxfp4_inputs(M, N, K, seed=22)
    A, B, (a, sa, b, sb) = _views(d, dev)
    C = torch.empty(M, N, dtype=torch.float16, device=dev)
    q.qgemm_mxfp4(A, B, C)
    A2 = q.qgemm_create_tensor(q.E2M1, a, sa + 1)
    C2 = torch.empty_like(C)
    q.qgemm_mxfp4(A2, B, C2)
    torch.cuda.synchronize()
    normal = C.abs() >= 2.0 ** -13
    assert torch.equal((C.float() * 2)[normal], C2.float()[normal])


def test_mxfp4_edge_cases(dev, orc):
    d = synth.mxfp4_inputs(64, 128, 128, seed=10)
    A, B, _ = _views(d, dev)
    # K = 0: the empty sum is zero
    A0 = q.qgemm_create_tensor(q.E2M1, torch.zeros(64, 16, dtype=torch.uint8, device=dev),
                               torch.zeros(64, 4, dtype=torch.uint8, device=dev), k=0)
    B0 = q.qgemm_create_tensor(q.E2M1, torch.zeros(128, 16, dtype=torch.uint8, device=dev),
                               torch.zeros(128, 4, dtype=torch.uint8, device=dev), k=0)
    C = torch.full((64, 128), 3.0, dtype=torch.float16, device=dev)
    q.qgemm_mxfp4(A0, B0, C)
    torch.cuda.synchronize()
    assert torch.all(C == 0)
    # M = 0: nothing happens
    q.qgemm_mxfp4(q.qgemm_tensor_slice(A, 0, 0, 0, 128), B, C[:0])
    # a 0xFF scale byte (NaN) poisons its row and only that row
    sa = d["sa"].clone()
    sa[7, 2] = 255
    An = q.qgemm_create_tensor(q.E2M1, d["a"].to(dev), sa.to(dev))
    Cn = torch.empty(64, 128, dtype=torch.float16, device=dev)
    q.qgemm_mxfp4(An, B, Cn)
    Cn = Cn.cpu()
    assert torch.isnan(Cn[7]).all()
    assert not torch.isnan(Cn[[0, 1, 2, 6, 8, 63]]).any()
    # the largest magnitudes: all +-6 at scale 2^0 gives exact integer sums
    K = 256
    six = torch.full((8, K // 2), 0x77, dtype=torch.uint8)          # +6 in both nibbles
    neg = torch.full((16, K // 2), 0xFF, dtype=torch.uint8)         # -6 in both nibbles
    s1 = torch.full((8, K // 32), 127, dtype=torch.uint8)
    s2 = torch.full((16, K // 32), 127, dtype=torch.uint8)
    Cx = torch.empty(8, 16, dtype=torch.float16, device=dev)
    q.qgemm_mxfp4(q.qgemm_create_tensor(q.E2M1, six.to(dev), s1.to(dev)),
                  q.qgemm_create_tensor(q.E2M1, neg.to(dev), s2.to(dev)), Cx)
    assert torch.all(Cx.cpu() == -36.0 * K)
    # wrong argument: error status, no launch
    with pytest.raises(q.QGemmError) as ei:
        q.qgemm_mxfp4(A, q.qgemm_tensor_slice(B, 0, 128, 0, 64), C)
    assert ei.value.name == "QGEMM_ERR_INVALID_ARG"


@pytest.mark.parametrize("accumulate,relu", [(True, False), (False, True), (True, True)])
def test_mxfp4_epilogue(dev, orc, accumulate, relu):
    M, N, K = 300, 520, 416
    d = synth.mxfp4_inputs(M, N, K, seed=M + N, row_variance=True)
    A, B, _ = _views(d, dev)
    res = _oracle(orc, d)
    old = (torch.randn((M, N), generator=synth.generator(16)) *
           (float(np.median(np.abs(res.C))) + 1e-3)).to(torch.float16)
    C = old.to(dev) if accumulate else torch.full((M, N), float("nan"), dtype=torch.float16,
                                                  device=dev)
    q.qgemm_mxfp4_ex(A, B, C, accumulate=accumulate, relu=relu)
    want = orc.epilogue(res, old.numpy() if accumulate else None, relu)
    _check(C, want, orc, what=f"mxfp4 epilogue acc={accumulate} relu={relu}")


def test_mxfp4_full_size_sampled(dev, orc):
    """8192^3 with per-row variance 10^U(-2,2): full GPU product, oracle on sampled rows."""
    d = synth.workload("mxfp4_8192")
    A, B, _ = _views(d, dev)
    C = torch.empty(8192, 8192, dtype=torch.float16, device=dev)
    q.qgemm_mxfp4(A, B, C)
    rows = np.sort(np.random.default_rng(1).choice(8192, 40, replace=False))
    rows = np.concatenate([[0, 127, 128, 8191], rows])
    res = _oracle(orc, d, rows)
    _check(C[torch.from_numpy(rows).to(dev)], res, orc, what="mxfp4 8192^3 sampled")
    for _ in range(2):                                                  # repeatable bit for bit
        C2 = torch.empty_like(C)
        q.qgemm_mxfp4(A, B, C2)
        assert torch.equal(C2.view(torch.int16), C.view(torch.int16))


def test_mxfp4_last_wave_half_tiles(dev, orc):
    """2048 x 3072: 76 whole pair tiles, then 20 left over as two 256 x 128 halves each; every
    element against the oracle, and the split columns bit-identical to whole tiles."""
    M, N, K = 2048, 3072, 512
    d = synth.mxfp4_inputs(M, N, K, seed=63, row_variance=True)
    A, B, _keep = _views(d, dev)
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
    q.qgemm_mxfp4(A, B, C)
    _check(C, _oracle(orc, d), orc, what="mxfp4 half tiles")
    Bs = q.qgemm_tensor_slice(B, 2304, 768, 0, K)
    Cs = torch.full((M, 768), float("nan"), dtype=torch.float16, device=dev)
    q.qgemm_mxfp4(A, Bs, Cs)
    torch.cuda.synchronize()
    assert torch.equal(Cs.view(torch.int16), C[:, 2304:].view(torch.int16))
