"""GPU parity of the custom-format int4 GEMM with fp16 block-32 scales (qgemm_w4a16_f16s) against
the oracle's M2-recipe product, through the C ABI.

The dequantised weights are checked bit for bit (an identity activation matrix makes C the
weights themselves: one product per output, exact in fp32 and in fp16); products are checked
element-wise with |C_gpu - C| <= 2e-3 * sum_k |a_mk w_nk| + 2^-24.
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


def test_fold_bit_exact_via_identity(dev, orc):
    """C = I W^T = the dequantised weights: every int4 value against scales spread over the
    fp16 range (subnormal, normal, large but finite after the multiply)."""
    K, N = 256, 300
    rng = np.random.default_rng(3)
    qv = rng.integers(-8, 8, size=(N, K))
    qv[:16, :16] = np.arange(-8, 8)[None, :]                     # every value appears
    mag = 2.0 ** rng.uniform(-24, 12, size=(N, K // 32))        # |q s| <= 8 * 2^12 < 65504
    sgn = np.where(rng.random((N, K // 32)) < 0.5, -1.0, 1.0)
    s = (mag * sgn).astype(np.float16)
    w = torch.from_numpy(((qv[:, 0::2] & 0xF) | ((qv[:, 1::2] & 0xF) << 4)).astype(np.uint8))
    A = torch.eye(K, dtype=torch.float16)
    C = torch.full((K, N), float("nan"), dtype=torch.float16, device=dev)
    q.qgemm_w4a16_f16s(A.to(dev), w.to(dev), torch.from_numpy(s).to(dev), C)
    torch.cuda.synchronize()
    assert q.qgemm_poll_device_error() == 0
    want = orc.dequant_int4_f16s(w.numpy(), s)                   # [N, K]
    got = C.float().cpu().numpy().astype(np.float64).T
    assert np.array_equal(got, want)


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (300, 520, 512), (96, 200, 256),
                                   (1, 64, 256), (257, 384, 1024), (640, 1000, 768)])
def test_w4a16_f16s_matches_oracle(dev, orc, M, N, K):
    d = synth.w4a16_f16s_inputs(M, N, K, seed=M + 7 * N + K)
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
    q.qgemm_w4a16_f16s(d["a"].to(dev), d["w"].to(dev), d["sw"].to(dev), C)
    res = orc.w4a16_f16s(d["a"].numpy(), d["w"].numpy(), d["sw"].numpy())
    _check(C, res, orc, what=f"w4a16 fp16-scale {M}x{N}x{K}")
    assert orc.cosine(C.float().cpu().numpy(), res.C) > 0.99999


def test_w4a16_f16s_padded_strides(dev, orc):
    """Padded rows for A, W, the scales and C; nothing written past N."""
    M, N, K = 200, 264, 512
    d = synth.w4a16_f16s_inputs(M, N, K, seed=44)
    a = torch.zeros(M, K + 64, dtype=torch.float16)
    a[:, :K] = d["a"]
    w = torch.zeros(N, K // 2 + 48, dtype=torch.uint8)
    w[:, :K // 2] = d["w"]
    s = torch.ones(N, K // 32 + 8, dtype=torch.float16)
    s[:, :K // 32] = d["sw"]
    Cbig = torch.full((M, N + 40), 7.0, dtype=torch.float16, device=dev)
    q.qgemm_w4a16_f16s(a.to(dev)[:, :K], w.to(dev)[:, :K // 2], s.to(dev)[:, :K // 32],
                       Cbig[:, :N])
    res = orc.w4a16_f16s(d["a"].numpy(), d["w"].numpy(), d["sw"].numpy())
    _check(Cbig[:, :N], res, orc, what="w4a16 fp16-scale strided")
    assert torch.all(Cbig[:, N:] == 7.0)


@pytest.mark.parametrize("accumulate,relu", [(True, False), (False, True), (True, True)])
def test_w4a16_f16s_epilogue(dev, orc, accumulate, relu):
    M, N, K = 300, 640, 512
    d = synth.w4a16_f16s_inputs(M, N, K, seed=45)
    res = orc.w4a16_f16s(d["a"].numpy(), d["w"].numpy(), d["sw"].numpy())
    old = (torch.randn((M, N), generator=synth.generator(17)) *
           (float(np.median(np.abs(res.C))) + 1e-3)).to(torch.float16)
    C = old.to(dev) if accumulate else torch.full((M, N), float("nan"), dtype=torch.float16,
                                                  device=dev)
    q.qgemm_w4a16_f16s_ex(d["a"].to(dev), d["w"].to(dev), d["sw"].to(dev), C,
                          accumulate=accumulate, relu=relu)
    want = orc.epilogue(res, old.numpy() if accumulate else None, relu)
    _check(C, want, orc, what=f"w4a16 fp16-scale epilogue acc={accumulate} relu={relu}")


def test_w4a16_f16s_edge_cases(dev):
    # K = 0 writes zeros
    C = torch.full((8, 16), 3.0, dtype=torch.float16, device=dev)
    a = torch.zeros(8, 8, dtype=torch.float16, device=dev)
    w = torch.zeros(16, 16, dtype=torch.uint8, device=dev)
    s = torch.zeros(16, 8, dtype=torch.float16, device=dev)
    q.load_library().qgemm_w4a16_f16s(q._ptr(a), 8, 8, q._ptr(w), 16, q._ptr(s), 8, 16, 0,
                                      q._ptr(C), 16, q._stream(None))
    torch.cuda.synchronize()
    assert torch.all(C == 0)
    # K not a multiple of 256: refused before launch
    d = synth.w4a16_f16s_inputs(16, 32, 288, seed=1)
    with pytest.raises(q.QGemmError) as ei:
        q.qgemm_w4a16_f16s(d["a"].to(dev), d["w"].to(dev), d["sw"].to(dev),
                           torch.empty(16, 32, dtype=torch.float16, device=dev))
    assert ei.value.name == "QGEMM_ERR_UNSUPPORTED_SHAPE"


def test_w4a16_f16s_full_size_sampled(dev, orc):
    """4096 x 14336 x 4096 (the prefill workload), oracle on sampled rows."""
    d = synth.workload("w4a16_f16s_prefill")
    C = torch.empty(4096, 14336, dtype=torch.float16, device=dev)
    q.qgemm_w4a16_f16s(d["a"].to(dev), d["w"].to(dev), d["sw"].to(dev), C)
    rows = np.sort(np.random.default_rng(2).choice(4096, 14, replace=False))
    rows = np.concatenate([[0, 4095], rows])
    res = orc.w4a16_f16s(d["a"].numpy(), d["w"].numpy(), d["sw"].numpy(), rows=rows)
    _check(C[torch.from_numpy(rows).to(dev)], res, orc, rows=None,
           what="w4a16 fp16-scale 4096x14336x4096 sampled")
    C2 = torch.empty_like(C)
    q.qgemm_w4a16_f16s(d["a"].to(dev), d["w"].to(dev), d["sw"].to(dev), C2)
    assert torch.equal(C2.view(torch.int16), C.view(torch.int16))     # repeatable bit for bit
