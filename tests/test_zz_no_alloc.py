"""qgemm_mxfp8_noalloc against qgemm_mxfp8, through the C ABI.

The no-allocation entry point exists for callers that cannot let a library allocate device
memory while they run -- a serving process whose own allocator owns all device memory, or a
latency-critical path that cannot risk an allocation that blocks or fails mid-request.  It keeps
the repacked scale planes in a fixed device buffer that every call shares, so these tests check
(1) two calls in a row, of different shapes, each give the product of the allocating entry
point within the parity tests' bound, the second call overwriting what the first left in the
buffer; and (2) a shape whose repacked scales do not fit the buffer is refused before anything is
launched.

The file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import block_scaled_quantized_tcgen05_gb300 as q
from block_scaled_quantized_tcgen05_gb300 import synth

pytestmark = pytest.mark.gpu

REL = 2e-3   # |C - C_ref| <= REL * sum_k |a_mk b_nk| + 2^-24, the parity tests' bound


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from block_scaled_quantized_tcgen05_gb300 import build
    build.build()
    q.load_library()
    q.qgemm_set_wait_timeout_ns(2_000_000_000)
    return torch.device("cuda:0")


def _views(M, N, K, seed, dev):
    d = synth.mxfp8_inputs(M, N, K, seed=seed, row_variance=True)
    A = q.qgemm_create_tensor(q.E4M3, d["a"].to(dev), d["sa"].to(dev))
    B = q.qgemm_create_tensor(q.E4M3, d["b"].to(dev), d["sb"].to(dev))
    return d, A, B


def test_noalloc_matches_allocating_entry_point_two_calls(dev, orc):
    # both shapes run on CTA pairs (M, N > 128) and so use the shared buffer; the second has a
    # ragged K and fewer row blocks, so it reads a different part of what the first one wrote
    cases = [(1000, 1536, 1024, 41), (640, 520, 416, 42)]
    runs = []
    for M, N, K, seed in cases:
        d, A, B = _views(M, N, K, seed, dev)
        ref = torch.empty(M, N, dtype=torch.float16, device=dev)
        q.qgemm_mxfp8(A, B, ref)
        out = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
        runs.append((d, A, B, ref, out))
    # one warm-up call: the first call on a device has the driver place the fixed array (CUDA
    # loads the library's modules lazily); from then on a call takes no device memory
    warm = torch.empty_like(runs[1][4])
    q.qgemm_mxfp8_noalloc(runs[1][1], runs[1][2], warm)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for d, A, B, ref, out in runs:           # the two no-alloc calls back to back on one stream
        q.qgemm_mxfp8_noalloc(A, B, out)
    torch.cuda.synchronize()
    assert q.qgemm_poll_device_error() == 0
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device free memory changed across the calls: {free0} -> {free1}"
    assert torch.cuda.memory_allocated() == alloc0
    for (M, N, K, _), (d, A, B, ref, out) in zip(cases, runs):
        res = orc.mxfp8(d["a"].numpy(), d["sa"].numpy(), d["b"].numpy(), d["sb"].numpy())
        got = out.float().cpu().numpy().astype(np.float64)
        want = ref.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all() and np.isfinite(want).all()
        bound = REL * res.D + 2.0 ** -24
        worst = float((np.abs(got - want) / bound).max())
        assert worst <= 1.0, f"no-alloc vs qgemm_mxfp8 at {M}x{N}x{K}: worst err/bound {worst}"
        ok, _, info = orc.within_tolerance(got, res, REL)
        assert ok, f"no-alloc vs oracle at {M}x{N}x{K}: {info}"


def test_noalloc_refuses_shapes_beyond_its_buffer(dev):
    # M = N = 16384, K = 8320 needs (128 + 128) * 65 * 512 bytes of repacked scales > 8 MiB.
    # Real buffers of that size back the views, so even a missed check could not read past them.
    M = N = 16384
    K = 8320
    a = torch.empty(M, K, dtype=torch.uint8, device=dev)
    sa = torch.full((M, K // 32), 127, dtype=torch.uint8, device=dev)
    A = q.qgemm_create_tensor(q.E4M3, a, sa)
    B = q.qgemm_create_tensor(q.E4M3, a, sa)
    C = torch.zeros(M, N, dtype=torch.float16, device=dev)
    with pytest.raises(q.QGemmError) as ei:
        q.qgemm_mxfp8_noalloc(A, B, C)
    assert ei.value.name == "QGEMM_ERR_UNSUPPORTED_SHAPE"
    assert "8388608" in str(ei.value) or "buffer" in str(ei.value)
    torch.cuda.synchronize()
    assert torch.count_nonzero(C).item() == 0        # nothing was launched
    del a, sa, C
    torch.cuda.empty_cache()


def test_noalloc_small_shapes_take_the_scratch_free_route(dev, orc):
    # M or N <= 128 runs the one-CTA kernel, which needs no scratch: same bits as qgemm_mxfp8
    for M, N, K, seed in [(128, 256, 128, 43), (96, 700, 320, 44)]:
        d, A, B = _views(M, N, K, seed, dev)
        ref = torch.empty(M, N, dtype=torch.float16, device=dev)
        out = torch.full((M, N), float("nan"), dtype=torch.float16, device=dev)
        q.qgemm_mxfp8(A, B, ref)
        q.qgemm_mxfp8_noalloc(A, B, out)
        torch.cuda.synchronize()
        assert q.qgemm_poll_device_error() == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        res = orc.mxfp8(d["a"].numpy(), d["sa"].numpy(), d["b"].numpy(), d["sb"].numpy())
        ok, _, info = orc.within_tolerance(out.float().cpu().numpy(), res, REL)
        assert ok, f"no-alloc one-CTA route at {M}x{N}x{K}: {info}"
