"""Split-K for decode-sized batches: the one-CTA MXFP8 and fp16 routes and the W4A16 CTA pairs,
through the C ABI.

An output of at most 128 rows on one side has few 128 x 256 tiles; when there are at most half as
many tiles as SMs, each tile's k range is shared out over S CTAs (whole 512-wide slices of K),
which write fp32 partial planes that a second kernel adds in split order before the one fp16
rounding.  Checked here against the oracle element by element -- ragged K, N <= 128 tiles, every
route by which the scale bytes reach shared memory, the fused epilogues, a NaN scale -- with the
split count the call must pick (read back through qgemm_mxfp8_scratch_bytes), bit-repeatability,
and agreement with the no-allocation entry point, which never splits.
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


def _plan(M, N, K, sms):
    """Split count and pooled bytes the library's rule gives on a GPU with `sms` SMs."""
    bn = 256 if N > 128 else 128
    tiles_n = -(-N // bn)
    tiles = -(-M // 128) * tiles_n
    units = -(-(-(-K // 128)) // 4)
    s = min(sms // tiles, units) if 2 * tiles <= sms else 1
    return s, (s * M * tiles_n * bn * 4 if s > 1 else 0)


def _views(d, dev, k0=0, K=None):
    A = q.qgemm_create_tensor(q.E4M3, d["a"].to(dev), d["sa"].to(dev))
    B = q.qgemm_create_tensor(q.E4M3, d["b"].to(dev), d["sb"].to(dev))
    if K is not None:
        A = q.qgemm_tensor_slice(A, 0, A.rows, k0, K)
        B = q.qgemm_tensor_slice(B, 0, B.rows, k0, K)
    return A, B


def _check(got, res, orc, what):
    assert q.qgemm_poll_device_error() == 0, f"{what}: device error word set"
    ok, _, info = orc.within_tolerance(got.float().cpu().numpy(), res, REL)
    assert ok, f"{what}: {info}"


@pytest.mark.parametrize("M,N,K", [
    (64, 4096, 4096),      # 16 tiles, 8 splits of one 512-slice each
    (1, 512, 4096),        # a single row
    (100, 1000, 2080),     # ragged last k-tile and column tile, uneven slices
    (128, 12288, 1024),    # 48 tiles, 2 splits
    (300, 96, 1536),       # N <= 128: 128 x 128 tiles (two accumulators), M over three tiles
    (96, 700, 8192),       # 16 splits of a long K
])
def test_split_k_matches_oracle(dev, orc, M, N, K):
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    S, nbytes = _plan(M, N, K, sms)
    assert S > 1, "the shape is meant to split"
    d = synth.mxfp8_inputs(M, N, K, seed=M + N + K, row_variance=True)
    A, B = _views(d, dev)
    assert q.qgemm_mxfp8_scratch_bytes(A, B) == nbytes
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
    q.qgemm_mxfp8(A, B, C)
    res = orc.mxfp8(d["a"].numpy(), d["sa"].numpy(), d["b"].numpy(), d["sb"].numpy())
    _check(C, res, orc, f"split-K {M}x{N}x{K} (S = {S})")
    C2 = torch.empty_like(C)
    q.qgemm_mxfp8(A, B, C2)
    torch.cuda.synchronize()
    assert torch.equal(C2.view(torch.int16), C.view(torch.int16))     # repeatable bit for bit


@pytest.mark.parametrize("k0", [128, 32, 0])
def test_split_k_scale_routes(dev, orc, k0):
    """A K window 128 elements in (scale rows 4-byte aligned: asynchronous 4-byte copies), one
    block in (1-byte aligned: byte loads), and none (16-byte aligned: TMA boxes)."""
    M, N, K = 64, 2048, 4096
    d = synth.mxfp8_inputs(M, N, K + 512, seed=200 + k0, row_variance=True)   # 144-byte scale rows
    A, B = _views(d, dev, k0, K)
    C = torch.empty(M, N, dtype=torch.float16, device=dev)
    q.qgemm_mxfp8(A, B, C)
    kb = slice(k0 // 32, (k0 + K) // 32)
    res = orc.mxfp8(d["a"][:, k0:k0 + K].numpy(), d["sa"][:, kb].numpy(),
                    d["b"][:, k0:k0 + K].numpy(), d["sb"][:, kb].numpy())
    _check(C, res, orc, f"split-K, K window at {k0}")


@pytest.mark.parametrize("accumulate,relu", [(True, False), (False, True), (True, True)])
def test_split_k_epilogue(dev, orc, accumulate, relu):
    M, N, K = 64, 1024, 4096
    d = synth.mxfp8_inputs(M, N, K, seed=7, row_variance=True)
    A, B = _views(d, dev)
    res = orc.mxfp8(d["a"].numpy(), d["sa"].numpy(), d["b"].numpy(), d["sb"].numpy())
    old = (torch.randn((M, N), generator=synth.generator(3)) *
           (float(np.median(np.abs(res.C))) + 1e-3)).to(torch.float16)
    C = old.to(dev) if accumulate else torch.full((M, N), float("nan"), dtype=torch.float16,
                                                  device=dev)
    q.qgemm_mxfp8_ex(A, B, C, accumulate=accumulate, relu=relu)
    _check(C, orc.epilogue(res, old.numpy() if accumulate else None, relu), orc,
           f"split-K epilogue acc={accumulate} relu={relu}")


def test_split_k_nan_scale_and_noalloc(dev, orc):
    """A NaN scale byte in one A block poisons exactly its row; the no-allocation entry point
    (one pass over K) agrees with the oracle as the split call does."""
    M, N, K = 64, 512, 4096
    d = synth.mxfp8_inputs(M, N, K, seed=11)
    d["sa"][3, 70] = 255
    A, B = _views(d, dev)
    C = torch.empty(M, N, dtype=torch.float16, device=dev)
    q.qgemm_mxfp8(A, B, C)
    res = orc.mxfp8(d["a"].numpy(), d["sa"].numpy(), d["b"].numpy(), d["sb"].numpy())
    _check(C, res, orc, "split-K with a NaN scale")
    Cn = C.float().cpu().numpy()
    assert np.isnan(Cn[3]).all() and np.isfinite(np.delete(Cn, 3, axis=0)).all()
    Cu = torch.empty_like(C)
    q.qgemm_mxfp8_noalloc(A, B, Cu)
    torch.cuda.synchronize()
    _check(Cu, res, orc, "one pass over K (no-alloc)")


def _f16_plan(M, N, K, sms):
    bn = 256 if N > 128 else 128
    tiles = -(-M // 128) * -(-N // bn)
    units = -(-(-(-K // 64)) // 8)
    return min(sms // tiles, units) if 2 * tiles <= sms else 1


@pytest.mark.parametrize("M,N,K", [(64, 4096, 4096), (1, 520, 2048), (100, 1000, 2080),
                                   (300, 96, 1536)])
def test_f16_split_k_matches_oracle(dev, orc, M, N, K):
    """The one-CTA fp16 route splits K the same way (fp32 partial planes, ordered reduction)."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    assert _f16_plan(M, N, K, sms) > 1, "the shape is meant to split"
    d = synth.f16_inputs(M, N, K, seed=M + 2 * N + K)
    a, b = d["a"].to(dev), d["b"].to(dev)
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
    q.gemm_f16(a, b, C)
    res = orc.gemm_f16(d["a"].numpy(), d["b"].numpy())
    _check(C, res, orc, f"fp16 split-K {M}x{N}x{K}")
    C2 = torch.empty_like(C)
    q.gemm_f16(a, b, C2)
    torch.cuda.synchronize()
    assert torch.equal(C2.view(torch.int16), C.view(torch.int16))


@pytest.mark.parametrize("accumulate,relu", [(True, True), (False, True)])
def test_f16_split_k_epilogue(dev, orc, accumulate, relu):
    M, N, K = 96, 768, 4096
    d = synth.f16_inputs(M, N, K, seed=5)
    res = orc.gemm_f16(d["a"].numpy(), d["b"].numpy())
    old = (torch.randn((M, N), generator=synth.generator(6)) *
           (float(np.median(np.abs(res.C))) + 1e-3)).to(torch.float16)
    C = old.to(dev) if accumulate else torch.full((M, N), float("nan"), dtype=torch.float16,
                                                  device=dev)
    q.gemm_f16_ex(d["a"].to(dev), d["b"].to(dev), C, accumulate=accumulate, relu=relu)
    _check(C, orc.epilogue(res, old.numpy() if accumulate else None, relu), orc,
           f"fp16 split-K epilogue acc={accumulate} relu={relu}")


# ---------------------------------------------------------------- W4A16 on CTA pairs, few tokens
# A few tokens against many weight rows fill few pair tiles; each tile's K is then split over up to
# pairs / tiles pairs (whole 512-wide slices), the partial planes added in order, and the outlier-row
# pass runs after that reduction.  Accumulating calls are not split (that pass needs the old C).
@pytest.mark.parametrize("M,N,K", [(64, 4096, 4096), (1, 1024, 2048), (100, 1000, 1024)])
def test_w4a16_split_k_matches_oracle(dev, orc, M, N, K):
    d = synth.w4a16_inputs(M, N, K, seed=M + N + K)
    W = q.qgemm_create_tensor(q.INT4, d["w"].to(dev), d["sw"].to(dev))
    a = d["a"].to(dev)
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
    q.qgemm_w4a16(a, W, C)
    res = orc.w4a16(d["a"].numpy(), d["w"].numpy(), d["sw"].numpy())
    _check(C, res, orc, f"w4a16 split-K {M}x{N}x{K}")
    C2 = torch.empty_like(C)
    q.qgemm_w4a16(a, W, C2)
    torch.cuda.synchronize()
    assert torch.equal(C2.view(torch.int16), C.view(torch.int16))


@pytest.mark.parametrize("accumulate,relu", [(False, False), (False, True), (True, True)])
def test_w4a16_split_k_every_scale_byte(dev, orc, accumulate, relu):
    """Every UE8M0 byte class, outlier rows included, on a 40-token batch (split unless the
    output is accumulated)."""
    M, N, K = 40, 600, 2048
    d = synth.w4a16_scale_extremes_inputs(M, N, K, seed=77)
    W = q.qgemm_create_tensor(q.INT4, d["w"].to(dev), d["sw"].to(dev))
    res = orc.w4a16(d["a"].numpy(), d["w"].numpy(), d["sw"].numpy())
    old = (torch.randn((M, N), generator=synth.generator(8)) * 4).to(torch.float16)
    C = old.to(dev) if accumulate else torch.full((M, N), float("nan"), dtype=torch.float16,
                                                  device=dev)
    q.qgemm_w4a16_ex(d["a"].to(dev), W, C, accumulate=accumulate, relu=relu)
    if accumulate or relu:
        res = orc.epilogue(res, old.numpy() if accumulate else None, relu=relu)
    _check(C, res, orc, f"w4a16 split-K extremes acc={accumulate} relu={relu}")


@pytest.mark.parametrize("M,N,K", [(64, 1024, 2048), (40, 1000, 2304)])
def test_w4a16_f16s_split_k(dev, orc, M, N, K):
    """fp16 scales (4 k-tiles per scale group): K = 2304 leaves a last slice of four k-tiles."""
    d = synth.w4a16_f16s_inputs(M, N, K, seed=9 + K)
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
    q.qgemm_w4a16_f16s(d["a"].to(dev), d["w"].to(dev), d["sw"].to(dev), C)
    _check(C, orc.w4a16_f16s(d["a"].numpy(), d["w"].numpy(), d["sw"].numpy()), orc,
           f"w4a16 fp16 scales split-K {M}x{N}x{K}")
