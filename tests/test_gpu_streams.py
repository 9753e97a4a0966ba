"""Calls on several streams at once, through the C ABI: each result must equal, bit for bit, the
same call run alone.  Nothing a call keeps between launches (pooled scale scratch, the attention
workspace and its flags, the per-device context) may leak into another call that overlaps it.
"""
import pytest
import torch

import block_scaled_quantized_tcgen05_gb300 as q
from block_scaled_quantized_tcgen05_gb300 import synth

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


def test_overlapping_calls_on_streams_match_serial_calls(dev):
    # two CTA-pair calls (pooled scale scratch) and one small-M call whose K is split over CTAs
    # (pooled partial planes)
    mx = [synth.mxfp8_inputs(1024, 768, 1024, seed=s, row_variance=True) for s in (1, 2)]
    mx.append(synth.mxfp8_inputs(64, 768, 4096, seed=9, row_variance=True))
    f16 = synth.f16_inputs(768, 1024, 512, seed=3)
    w8 = synth.w8_inputs(9, 4096, 2048, seed=4)
    w4 = synth.w4a16_inputs(384, 512, 1024, seed=5)
    # attention whose key tiles are shared out in ranges that cut units (tails and heads merged
    # through a per-call workspace and flags; cooperative launches)
    at = [synth.attention_inputs(8, 512, 1000, 128, seed=6, q_std=2.0),
          synth.attention_inputs(3, 200, 2048, 128, seed=7)]

    def views():
        out = []
        for d in mx:
            A = q.qgemm_create_tensor(q.E4M3, d["a"].to(dev), d["sa"].to(dev))
            B = q.qgemm_create_tensor(q.E4M3, d["b"].to(dev), d["sb"].to(dev))
            out.append((A, B))
        return out

    mxv = views()
    fa, fb = f16["a"].to(dev), f16["b"].to(dev)
    W8 = q.qgemm_create_tensor(q.INT8, w8["w"].to(dev), w8["sw"].to(dev))
    x8 = w8["x"].to(dev)
    W4 = q.qgemm_create_tensor(q.INT4, w4["w"].to(dev), w4["sw"].to(dev))
    a4 = w4["a"].to(dev)
    atd = [tuple(d[k].to(dev) for k in ("q", "k", "v")) + (d["scale"],) for d in at]

    def run(streams):
        outs = [torch.empty(d["a"].shape[0], 768, dtype=torch.float16, device=dev) for d in mx]
        cf = torch.empty(768, 1024, dtype=torch.float16, device=dev)
        y8 = torch.empty(9, 4096, dtype=torch.float16, device=dev)
        c4 = torch.empty(384, 512, dtype=torch.float16, device=dev)
        ao = [torch.empty_like(t[0]) for t in atd]
        calls = [lambda s, i=i: q.qgemm_mxfp8(mxv[i][0], mxv[i][1], outs[i], stream=s)
                 for i in range(len(mxv))]
        calls += [lambda s: q.gemm_f16(fa, fb, cf, stream=s),
                  lambda s: q.qgemm_w8_gemv(x8, W8, y8, stream=s),
                  lambda s: q.qgemm_w4a16(a4, W4, c4, stream=s)]
        calls += [lambda s, i=i: q.qgemm_attention(atd[i][0], atd[i][1], atd[i][2], ao[i],
                                                   scale=atd[i][3], stream=s) for i in range(2)]
        torch.cuda.synchronize()
        for rep in range(3):
            for i, call in enumerate(calls):
                call(streams[i % len(streams)])
        torch.cuda.synchronize()
        return [t.clone() for t in outs + [cf, y8, c4] + ao]

    serial = run([torch.cuda.current_stream()])
    side = [torch.cuda.Stream() for _ in range(7)]
    for _ in range(3):
        overlapped = run(side)
        for s, o in zip(serial, overlapped):
            assert torch.equal(s.view(torch.int16), o.view(torch.int16))
    assert q.qgemm_poll_device_error() == 0
