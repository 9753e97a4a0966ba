"""qgemm_mxfp8_host: operands and output in host memory, through the C ABI.

The chunked, overlapped call must give exactly the bits of qgemm_mxfp8 on device copies of the
same operands (the row chunks start on pair-tile boundaries, so every output element is formed
by the same arithmetic) and match the oracle within the parity bound.
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


def _host_views(d):
    a, sa, b, sb = (d[k].pin_memory() for k in ("a", "sa", "b", "sb"))
    return q.qgemm_create_tensor(q.E4M3, a, sa), q.qgemm_create_tensor(q.E4M3, b, sb), (a, sa, b, sb)


def _device_ref(d, dev):
    a, sa, b, sb = (d[k].to(dev) for k in ("a", "sa", "b", "sb"))
    C = torch.empty(d["a"].shape[0], d["b"].shape[0], dtype=torch.float16, device=dev)
    q.qgemm_mxfp8(q.qgemm_create_tensor(q.E4M3, a, sa), q.qgemm_create_tensor(q.E4M3, b, sb), C)
    return C.cpu()


# the last shape splits K over eight CTAs on the one-CTA route (A is a single row chunk): the host
# call must take the same route and sum order as the device call
@pytest.mark.parametrize("M,N,K", [(300, 520, 416), (1000, 1536, 1024), (64, 96, 128), (64, 2048, 4096)])
def test_host_call_matches_device_call_and_oracle(dev, orc, M, N, K):
    d = synth.mxfp8_inputs(M, N, K, seed=M + N + 3, row_variance=True)
    A, B, _ = _host_views(d)
    C = torch.full((M, N), float("nan"), dtype=torch.float16).pin_memory()
    q.qgemm_mxfp8_host(A, B, C)
    torch.cuda.synchronize()
    assert q.qgemm_poll_device_error() == 0
    assert torch.equal(C, _device_ref(d, dev))
    res = orc.mxfp8(d["a"].numpy(), d["sa"].numpy(), d["b"].numpy(), d["sb"].numpy())
    ok, _, info = orc.within_tolerance(C.float().numpy(), res, REL)
    assert ok, info


def test_host_calls_in_flight_on_two_streams(dev, orc):
    """Two calls on two streams overlap (and use the two buffer sets); a third, larger call grows
    a set; strided host views and a padded host C."""
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    d1 = synth.mxfp8_inputs(1024, 768, 512, seed=91, row_variance=True)
    d2 = synth.mxfp8_inputs(520, 1300, 384, seed=92, row_variance=True)
    A1, B1, _ = _host_views(d1)
    # d2's A lives in a wider host buffer (row stride K + 64), C2 has 8 columns of padding
    a2 = torch.zeros(520, 384 + 64, dtype=torch.uint8)
    a2[:, :384] = d2["a"]
    a2 = a2.pin_memory()
    sa2 = d2["sa"].pin_memory()
    A2 = q.qgemm_create_tensor(q.E4M3, a2[:, :384], sa2)
    B2 = q.qgemm_create_tensor(q.E4M3, d2["b"].pin_memory(), d2["sb"].pin_memory())
    C1 = torch.empty(1024, 768, dtype=torch.float16).pin_memory()
    C2big = torch.full((520, 1308), 5.0, dtype=torch.float16).pin_memory()
    q.qgemm_mxfp8_host(A1, B1, C1, stream=s1)
    q.qgemm_mxfp8_host(A2, B2, C2big[:, :1300], stream=s2)
    d3 = synth.mxfp8_inputs(2048, 1024, 1024, seed=93, row_variance=True)
    A3, B3, _ = _host_views(d3)
    C3 = torch.empty(2048, 1024, dtype=torch.float16).pin_memory()
    q.qgemm_mxfp8_host(A3, B3, C3, stream=s1)
    torch.cuda.synchronize()
    assert q.qgemm_poll_device_error() == 0
    assert torch.equal(C1, _device_ref(d1, dev))
    assert torch.equal(C2big[:, :1300], _device_ref(d2, dev))
    assert torch.all(C2big[:, 1300:] == 5.0)
    assert torch.equal(C3, _device_ref(d3, dev))


def test_host_call_edge_cases(dev):
    # K = 0: zeros
    a0 = torch.zeros(64, 16, dtype=torch.uint8).pin_memory()
    s0 = torch.zeros(64, 1, dtype=torch.uint8).pin_memory()
    A0 = q.qgemm_create_tensor(q.E4M3, a0, s0, k=0)
    B0 = q.qgemm_create_tensor(q.E4M3, a0, s0, k=0)
    C = torch.full((64, 64), 3.0, dtype=torch.float16).pin_memory()
    q.qgemm_mxfp8_host(A0, B0, C)
    torch.cuda.synchronize()
    assert torch.all(C == 0)
    # wrong dtype: refused before anything is enqueued
    d = synth.w8_inputs(4, 64, 128, seed=2)
    W = q.qgemm_create_tensor(q.INT8, d["w"], d["sw"])
    with pytest.raises(q.QGemmError) as ei:
        q.qgemm_mxfp8_host(W, W, torch.empty(64, 64, dtype=torch.float16))
    assert ei.value.name == "QGEMM_ERR_UNSUPPORTED_DTYPE"
