"""W4A16 over the whole UE8M0 byte range, on every kernel route, against the oracle.

The product is defined for every scale byte ("TensorOps: quantized matmul ...", section "M2 =
block-32 fp16 scaling": each 32-block of int4 weights times its block scale, then the product
with the activations; section "Kernel-phase findings": the scale is an E8M0 power of two, 255
being NaN).  The weights here put bytes 0, 1, 60, 102, 140..146, 180, 254 and 255 into rows
(with nonzero and with all-zero weights) and across rows; the activations are scaled per block
so that the outputs stay far above the fp16 output quantum and below its overflow, except for
the rows built to overflow or to be NaN.  Every output element is compared with the fp64 oracle
under the element-wise tolerance, for the plain store and the three fused epilogues.
"""
import numpy as np
import pytest
import torch

import block_scaled_quantized_tcgen05_gb300 as q
from block_scaled_quantized_tcgen05_gb300 import synth

pytestmark = pytest.mark.gpu

REL = 2e-3

# (name, M, N, K, scale-row padding in bytes): which kernel runs is decided by the shape and
# the scale rows' alignment -- CTA pairs (N > 128, K % 512 == 0, 16-byte scale rows; any M, a
# few tokens included), the one-CTA TMA route (the same with N <= 128), and the one-CTA cp.async
# route (K % 512 != 0)
# with 4-byte scale words or, for scale rows 21 bytes apart, byte loads.
ROUTES = [
    ("pair", 300, 600, 1024, 0),
    ("pair_many_ctas", 1100, 600, 512, 0),
    ("pair_few_tokens", 40, 600, 1024, 0),
    ("tma_one_cta", 300, 120, 1024, 0),
    ("cp_async_word_scales", 200, 300, 640, 0),
    ("cp_async_byte_scales", 200, 300, 640, 1),
]
EPILOGUES = [(False, False), (False, True), (True, False), (True, True)]


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from block_scaled_quantized_tcgen05_gb300 import build
    build.build()
    q.load_library()
    q.qgemm_set_wait_timeout_ns(2_000_000_000)
    return torch.device("cuda:0")


def _inputs(M, N, K, pad, seed, dev):
    d = synth.w4a16_scale_extremes_inputs(M, N, K, seed=seed)
    nblk = K // 32
    if pad:
        full = torch.full((N, nblk + pad), 127, dtype=torch.uint8)
        full[:, :nblk] = d["sw"]
        sv = full.to(dev)[:, :nblk]
    else:
        sv = d["sw"].to(dev)
    return d, q.qgemm_create_tensor(q.INT4, d["w"].to(dev), sv), sv


@pytest.mark.parametrize("accumulate,relu", EPILOGUES)
@pytest.mark.parametrize("name,M,N,K,pad", ROUTES)
def test_w4a16_every_scale_byte(dev, orc, name, M, N, K, pad, accumulate, relu):
    d, W, _sv = _inputs(M, N, K, pad, seed=M + N + K + pad, dev=dev)
    a = d["a"].to(dev)
    g = synth.generator(17)
    c_old = (torch.randn(M, N, generator=g) * 4).to(torch.float16)
    C = c_old.to(dev) if accumulate else torch.full((M, N), float("nan"), dtype=torch.float16,
                                                    device=dev)
    q.qgemm_w4a16_ex(a, W, C, accumulate=accumulate, relu=relu)
    code = q.qgemm_poll_device_error()
    assert code == 0, f"a device wait timed out (error word {code:#x})"
    res = orc.w4a16(d["a"].numpy(), d["w"].numpy(), d["sw"].numpy())
    if accumulate or relu:
        res = orc.epilogue(res, c_old.numpy() if accumulate else None, relu=relu)
    got = C.float().cpu().numpy()
    ok, worst, info = orc.within_tolerance(got, res, REL)
    kind = d["kind"].numpy()
    if not ok:
        bad_cols = np.unique(np.nonzero(~np.isclose(got, res.f16.astype(np.float64),
                                                    equal_nan=True))[1])
        raise AssertionError(f"{name} acc={accumulate} relu={relu}: {info}; row kinds of the "
                             f"differing columns: {np.bincount(kind[bad_cols], minlength=9)}")
    # the inputs did what they are for: NaN rows, overflowing rows, small outputs far above
    # the fp16 quantum where the low scale bytes carry the sum
    ref = res.f16.astype(np.float64)
    if not relu:
        assert np.isnan(ref[:, kind == 5]).all() and np.isnan(ref[:, kind == 6]).all()
        if not accumulate:
            assert np.isinf(ref[:, kind == 7]).all()
            for k_ in (2, 8):
                assert np.median(np.abs(ref[:, kind == k_])) > 1000 * 2.0 ** -24


@pytest.mark.parametrize("name,M,N,K,pad", ROUTES[:4])
def test_w4a16_every_scale_byte_repeatable(dev, name, M, N, K, pad):
    """Outlier rows are summed in a fixed order: two calls give the same bits."""
    d, W, _sv = _inputs(M, N, K, pad, seed=5 * M + N, dev=dev)
    a = d["a"].to(dev)
    C1 = torch.empty(M, N, dtype=torch.float16, device=dev)
    C2 = torch.empty(M, N, dtype=torch.float16, device=dev)
    q.qgemm_w4a16(a, W, C1)
    q.qgemm_w4a16(a, W, C2)
    torch.cuda.synchronize()
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))
