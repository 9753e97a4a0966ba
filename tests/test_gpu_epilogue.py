"""GPU parity of the fused output epilogue, C = relu?(A*B [+ C_old]), through the C ABI.

Every GEMM family on each of its kernel routes (CTA pairs for large M and N, one CTA per tile
otherwise, the W4A16 routes by scale alignment and K), and the decode GEMV, against the oracle's
epilogue: the exact product plus C_old in fp64, ReLU, one fp16 rounding; tolerance
|C_gpu - C| <= 2e-3 * (sum |a b| + |C_old|) + 2^-24.
"""
import numpy as np
import pytest
import torch

import block_scaled_quantized_tcgen05_gb300 as q
from block_scaled_quantized_tcgen05_gb300 import synth

pytestmark = pytest.mark.gpu

REL = 2e-3
MODES = [(True, False), (False, True), (True, True)]   # (accumulate, relu)


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from block_scaled_quantized_tcgen05_gb300 import build
    build.build()
    q.load_library()
    q.qgemm_set_wait_timeout_ns(2_000_000_000)
    return torch.device("cuda:0")


def _old(shape, seed, scale):
    """C_old: seeded fp16 values of the product's magnitude, about half of them negative."""
    return (torch.randn(shape, generator=synth.generator(seed)) * scale).to(torch.float16)


def _check(got, res, orc, what):
    assert q.qgemm_poll_device_error() == 0, f"{what}: a device wait timed out"
    ok, _, info = orc.within_tolerance(got.float().cpu().numpy(), res, REL)
    assert ok, f"{what}: {info}"


@pytest.mark.parametrize("accumulate,relu", MODES)
@pytest.mark.parametrize("M,N,K", [(300, 520, 416), (96, 200, 256)])
def test_mxfp8_epilogue(dev, orc, M, N, K, accumulate, relu):
    d = synth.mxfp8_inputs(M, N, K, seed=M + N, row_variance=True)
    A = q.qgemm_create_tensor(q.E4M3, d["a"].to(dev), d["sa"].to(dev))
    B = q.qgemm_create_tensor(q.E4M3, d["b"].to(dev), d["sb"].to(dev))
    res = orc.mxfp8(d["a"].numpy(), d["sa"].numpy(), d["b"].numpy(), d["sb"].numpy())
    old = _old((M, N), 11, float(np.median(np.abs(res.C))) + 1e-3)
    C = old.to(dev) if accumulate else torch.full((M, N), float("nan"), dtype=torch.float16,
                                                  device=dev)
    q.qgemm_mxfp8_ex(A, B, C, accumulate=accumulate, relu=relu)
    want = orc.epilogue(res, old.numpy() if accumulate else None, relu)
    _check(C, want, orc, f"mxfp8 {M}x{N}x{K} acc={accumulate} relu={relu}")


@pytest.mark.parametrize("accumulate,relu", MODES)
@pytest.mark.parametrize("M,N,K", [(384, 512, 256), (96, 64, 128)])
def test_f16_epilogue(dev, orc, M, N, K, accumulate, relu):
    d = synth.f16_inputs(M, N, K, seed=M + 2 * N)
    res = orc.gemm_f16(d["a"].numpy(), d["b"].numpy())
    old = _old((M, N), 12, float(np.median(np.abs(res.C))) + 1e-3)
    C = old.to(dev) if accumulate else torch.empty(M, N, dtype=torch.float16, device=dev)
    q.gemm_f16_ex(d["a"].to(dev), d["b"].to(dev), C, accumulate=accumulate, relu=relu)
    want = orc.epilogue(res, old.numpy() if accumulate else None, relu)
    _check(C, want, orc, f"f16 {M}x{N}x{K} acc={accumulate} relu={relu}")


@pytest.mark.parametrize("accumulate,relu", MODES)
@pytest.mark.parametrize("M,N,K", [(300, 640, 1536), (128, 300, 512), (128, 256, 64)])
def test_w4a16_epilogue(dev, orc, M, N, K, accumulate, relu):
    # (300, 640, 1536): CTA pairs with the weights in TMEM; (128, 300, 512): one CTA, TMA-fed
    # scales; (128, 256, 64): one CTA, scales by cp.async
    d = synth.w4a16_inputs(M, N, K, seed=M + 5 * N)
    W = q.qgemm_create_tensor(q.INT4, d["w"].to(dev), d["sw"].to(dev))
    res = orc.w4a16(d["a"].numpy(), d["w"].numpy(), d["sw"].numpy())
    old = _old((M, N), 13, float(np.median(np.abs(res.C))) + 1e-3)
    C = old.to(dev) if accumulate else torch.empty(M, N, dtype=torch.float16, device=dev)
    q.qgemm_w4a16_ex(d["a"].to(dev), W, C, accumulate=accumulate, relu=relu)
    want = orc.epilogue(res, old.numpy() if accumulate else None, relu)
    _check(C, want, orc, f"w4a16 {M}x{N}x{K} acc={accumulate} relu={relu}")


@pytest.mark.parametrize("accumulate,relu", MODES)
@pytest.mark.parametrize("M", [1, 9])
def test_w8_gemv_epilogue(dev, orc, M, accumulate, relu):
    N, K = 1000, 2048
    d = synth.w8_inputs(M, N, K, seed=M + 40)
    W = q.qgemm_create_tensor(q.INT8, d["w"].to(dev), d["sw"].to(dev))
    res = orc.w8_gemv(d["x"].numpy(), d["w"].numpy(), d["sw"].numpy())
    old = _old((M, N), 14, float(np.median(np.abs(res.C))) + 1e-3)
    Y = old.to(dev) if accumulate else torch.empty(M, N, dtype=torch.float16, device=dev)
    q.qgemm_w8_gemv_ex(d["x"].to(dev), W, Y, accumulate=accumulate, relu=relu)
    want = orc.epilogue(res, old.numpy() if accumulate else None, relu)
    _check(Y, want, orc, f"w8 gemv M={M} acc={accumulate} relu={relu}")


def test_epilogue_empty_reduction(dev):
    """K = 0: accumulate leaves C_old (ReLU applied), plain mode writes zeros."""
    old = _old((64, 96), 15, 1.0).to(dev)
    A0 = q.qgemm_create_tensor(q.E4M3, torch.zeros(64, 16, dtype=torch.uint8, device=dev),
                               torch.zeros(64, 4, dtype=torch.uint8, device=dev), k=0)
    B0 = q.qgemm_create_tensor(q.E4M3, torch.zeros(96, 16, dtype=torch.uint8, device=dev),
                               torch.zeros(96, 4, dtype=torch.uint8, device=dev), k=0)
    C = old.clone()
    q.qgemm_mxfp8_ex(A0, B0, C, accumulate=True, relu=False)
    torch.cuda.synchronize()
    assert torch.equal(C, old)
    q.qgemm_mxfp8_ex(A0, B0, C, accumulate=True, relu=True)
    torch.cuda.synchronize()
    assert torch.equal(C, torch.clamp(old, min=0))
    q.qgemm_mxfp8_ex(A0, B0, C, accumulate=False, relu=True)
    torch.cuda.synchronize()
    assert torch.all(C == 0)
