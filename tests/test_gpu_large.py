"""Operands larger than 2^31 bytes, through the C ABI: every byte offset past 2 GiB must be formed
in 64 bits.  The data are uniform random bytes (E4M3 NaN codes replaced), so nothing but the
addressing is under test; the oracle checks sampled outputs, including the last rows.
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


def _bytes(shape, seed, lo=0, hi=256):
    return torch.randint(lo, hi, shape, generator=synth.generator(seed), dtype=torch.uint8)


def test_w8_gemv_weights_beyond_2gib(dev, orc):
    M, N, K = 3, 266240, 8192                      # 2.18e9 weight bytes
    assert N * K > 2 ** 31
    w = _bytes((N, K), 11)
    sw = _bytes((N, K // 32), 12, 100, 141)
    x = synth.normal((M, K), synth.generator(13)).to(torch.float16)
    W = q.qgemm_create_tensor(q.INT8, w.to(dev), sw.to(dev))
    Y = torch.empty(M, N, dtype=torch.float16, device=dev)
    q.qgemm_w8_gemv(x.to(dev), W, Y)
    assert q.qgemm_poll_device_error() == 0
    cols = np.concatenate([[0, 262143, 262144, N - 1], np.sort(np.random.default_rng(5).choice(N, 60, replace=False))])
    res = orc.w8_gemv(x.numpy(), w.numpy()[cols], sw.numpy()[cols])
    ok, _, info = orc.within_tolerance(Y[:, torch.from_numpy(cols).to(dev)].float().cpu().numpy(), res, REL)
    assert ok, info


def test_mxfp8_operand_beyond_2gib(dev, orc):
    M, N, K = 66048, 256, 32768                    # A: 2.16e9 bytes
    assert M * K > 2 ** 31
    a = _bytes((M, K), 21)
    a[(a & 0x7F) == 0x7F] -= 1                     # no NaN codes (0x7f, 0xff -> 0x7e, 0xfe)
    b = _bytes((N, K), 22)
    b[(b & 0x7F) == 0x7F] -= 1
    sa = _bytes((M, K // 32), 23, 120, 135)
    sb = _bytes((N, K // 32), 24, 120, 135)
    A = q.qgemm_create_tensor(q.E4M3, a.to(dev), sa.to(dev))
    B = q.qgemm_create_tensor(q.E4M3, b.to(dev), sb.to(dev))
    C = torch.empty(M, N, dtype=torch.float16, device=dev)
    q.qgemm_mxfp8(A, B, C)
    assert q.qgemm_poll_device_error() == 0
    rows = np.concatenate([[0, 65535 - 256, M - 1], np.sort(np.random.default_rng(6).choice(M, 29, replace=False))])
    res = orc.mxfp8(a.numpy()[rows], sa.numpy()[rows], b.numpy(), sb.numpy())
    ok, _, info = orc.within_tolerance(C[torch.from_numpy(rows).to(dev)].float().cpu().numpy(), res, REL)
    assert ok, info
