"""The CUDA path against the golden fixtures under tests/golden/, through the C ABI.

The hand-worked MXFP8 products are exact in fp32 whatever the summation order, so the kernel's
fp16 output must match the fixture bit for bit.  The validation table's printed cosine similarity
(1.000000) is checked for the library's kernels on the pages' o-proj shape, beside the element-wise
oracle tolerance.
"""
import pytest
import torch

import block_scaled_quantized_tcgen05_gb300 as q
from block_scaled_quantized_tcgen05_gb300 import synth

from test_golden import _lines, mxfp8_cases, validation_case, validation_int_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from block_scaled_quantized_tcgen05_gb300 import build
    build.build()
    q.load_library()
    q.qgemm_set_wait_timeout_ns(2_000_000_000)
    return torch.device("cuda:0")


def test_mxfp8_hand_worked_bits(dev):
    n = 0
    for name, A, SA, B, SB, _, _, bits in mxfp8_cases():
        ta = q.qgemm_create_tensor(q.E4M3, torch.from_numpy(A).to(dev), torch.from_numpy(SA).to(dev))
        tb = q.qgemm_create_tensor(q.E4M3, torch.from_numpy(B).to(dev), torch.from_numpy(SB).to(dev))
        C = torch.full((1, 1), 7.0, dtype=torch.float16, device=dev)
        q.qgemm_mxfp8(ta, tb, C)
        got = C.cpu()
        if bits is None:
            assert torch.isnan(got).all(), name
        else:
            assert int(got.view(torch.int16)[0, 0]) & 0xFFFF == bits, name
        n += 1
    assert q.qgemm_poll_device_error() == 0
    assert n >= 15


@pytest.mark.parametrize("kernel", ["M0", "M1a", "M1b", "M2"])
def test_validation_table_on_gpu(dev, orc, kernel):
    row = [r for r in ([x.strip() for x in line.split("|")] for line in _lines("validation_cos_sim.txt"))
           if r[0] == kernel][0]
    M, K, N = (int(x) for x in row[2].split())
    res, ref = validation_case(orc, kernel, M, K, N)
    g = synth.generator(7)
    x = synth.normal((M, K), g).to(torch.float16)
    w = synth.normal((N, K), g, std=0.02)
    C = torch.empty(M, N, dtype=torch.float16, device=dev)
    if kernel == "M0":
        q.gemm_f16(x.to(dev), w.to(torch.float16).t().contiguous().to(dev), C)
    elif kernel == "M1a":
        d = validation_int_weights(w, 127)
        W = q.qgemm_create_tensor(q.INT8, d["q"].view(torch.uint8).to(dev), d["s"].to(dev))
        xd = x.to(dev)
        for m0 in range(0, M, 16):                     # the decode GEMV takes up to 16 rows a call
            q.qgemm_w8_gemv(xd[m0:m0 + 16], W, C[m0:m0 + 16])
    elif kernel == "M1b":
        d = validation_int_weights(w, 7)
        W = q.qgemm_create_tensor(q.INT4, synth.pack_int4(d["q"]).to(dev), d["s"].to(dev))
        q.qgemm_w4a16(x.to(dev), W, C)
    else:
        d = synth.w4a16_f16s_inputs(M, N, K, 7)
        q.qgemm_w4a16_f16s(d["a"].to(dev), d["w"].to(dev), d["sw"].to(dev), C)
    assert q.qgemm_poll_device_error() == 0
    got = C.float().cpu().numpy()
    assert f"{orc.cosine(got, ref):.6f}" == row[3], kernel
    ok, _, info = orc.within_tolerance(got, res, 2e-3)
    assert ok, f"{kernel}: {info}"
