"""The debug build (QGEMM_DEBUG): every kernel checks its own index arithmetic -- TMA coordinates,
offsets into the repacked scale planes and the attention workspace, the schedule of the attention
key-tile ranges -- and reports a failed check as bit 32 of the device error word instead of making
the access.  It stands in for a memory sanitizer: this test runs every kernel route of the debug
library on small and ragged shapes, in a child process started with QGEMM_DEBUG=1 (the binding
then loads libqgemm_debug.so), checks each result against the oracle and requires a clean error
word after each call.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import os, sys
sys.path.insert(0, os.environ["QG_ROOT"])
import numpy as np
import torch
from block_scaled_quantized_tcgen05_gb300 import build
build.build(debug=True)
import __graft_entry__ as g
import block_scaled_quantized_tcgen05_gb300 as q
import oracle
from block_scaled_quantized_tcgen05_gb300 import synth

assert os.path.basename(q.library_path()) == "libqgemm_debug.so", q.library_path()
assert q.qgemm_debug_build(), "the loaded library was not compiled with QGEMM_DEBUG"
g.smoke()   # every hot-path route against the oracle; raises on a non-zero error word
dev = torch.device("cuda:0")


def clean(what):
    torch.cuda.synchronize()
    word = q.qgemm_poll_device_error()
    if word != 0:
        raise RuntimeError(f"{what}: device error word {word:#x}")


def close(what, got, ref):
    ok, _, info = oracle.within_tolerance(got.float().cpu().numpy().reshape(ref.C.shape), ref)
    if not ok:
        raise RuntimeError(f"{what}: {info}")


# fp16 one-CTA route (M <= 128) and MXFP8 with a K that ends inside a k-tile, both routes
df = synth.f16_inputs(100, 200, 64, seed=31)
Cf = torch.empty(100, 200, dtype=torch.float16, device=dev)
q.gemm_f16(df["a"].to(dev), df["b"].to(dev), Cf)
clean("fp16 one-CTA")
close("fp16 one-CTA", Cf, oracle.gemm_f16(df["a"].numpy(), df["b"].numpy()))
for (M, N, K) in ((300, 520, 224), (100, 136, 224)):
    d = synth.mxfp8_inputs(M, N, K, seed=M + K)
    A = q.qgemm_create_tensor(q.E4M3, d["a"].to(dev), d["sa"].to(dev))
    B = q.qgemm_create_tensor(q.E4M3, d["b"].to(dev), d["sb"].to(dev))
    C = torch.empty(M, N, dtype=torch.float16, device=dev)
    q.qgemm_mxfp8(A, B, C)
    clean(f"mxfp8 {M}x{N}x{K}")
    close(f"mxfp8 {M}x{N}x{K}", C, oracle.mxfp8(d["a"].numpy(), d["sa"].numpy(),
                                                 d["b"].numpy(), d["sb"].numpy()))
# fp16 one-CTA route with K split over CTAs (ragged last k-tile)
df = synth.f16_inputs(64, 1000, 2080, seed=32)
Cf = torch.empty(64, 1000, dtype=torch.float16, device=dev)
q.gemm_f16(df["a"].to(dev), df["b"].to(dev), Cf)
clean("fp16 split-K")
close("fp16 split-K", Cf, oracle.gemm_f16(df["a"].numpy(), df["b"].numpy()))
# MXFP8 one-CTA route with K split over CTAs (partial planes, then the ordered reduction), with a
# K window that starts one scale byte in
for (M, N, K, k0) in ((64, 1000, 2080, 0), (40, 520, 1024, 32)):
    d = synth.mxfp8_inputs(M, N, K + k0, seed=M + K)
    A = q.qgemm_create_tensor(q.E4M3, d["a"].to(dev), d["sa"].to(dev))
    B = q.qgemm_create_tensor(q.E4M3, d["b"].to(dev), d["sb"].to(dev))
    A, B = q.qgemm_tensor_slice(A, 0, M, k0, K), q.qgemm_tensor_slice(B, 0, N, k0, K)
    assert q.qgemm_mxfp8_scratch_bytes(A, B) > 0, "meant to split K"
    C = torch.empty(M, N, dtype=torch.float16, device=dev)
    q.qgemm_mxfp8(A, B, C)
    clean(f"mxfp8 split-K {M}x{N}x{K}")
    kb = slice(k0 // 32, (k0 + K) // 32)
    close(f"mxfp8 split-K {M}x{N}x{K}", C,
          oracle.mxfp8(d["a"][:, k0:k0 + K].numpy(), d["sa"][:, kb].numpy(),
                       d["b"][:, k0:k0 + K].numpy(), d["sb"][:, kb].numpy()))
# W4A16 on CTA pairs with K split over four pairs (few tokens), outlier rows included
dw = synth.w4a16_scale_extremes_inputs(40, 1000, 2048, seed=34)
Ww = q.qgemm_create_tensor(q.INT4, dw["w"].to(dev), dw["sw"].to(dev))
Cw = torch.empty(40, 1000, dtype=torch.float16, device=dev)
q.qgemm_w4a16(dw["a"].to(dev), Ww, Cw)
clean("w4a16 split-K")
close("w4a16 split-K", Cw, oracle.w4a16(dw["a"].numpy(), dw["w"].numpy(), dw["sw"].numpy()))
# attention: a CTA with a tail first and a head last; one unit over eight CTAs
for (BH, Lq, Lk) in ((3, 200, 300), (1, 100, 4096)):
    d = synth.attention_inputs(BH, Lq, Lk, 128, seed=BH + Lk, q_std=2.0)
    Q, K_, V = (d[k].to(dev) for k in ("q", "k", "v"))
    O = torch.empty_like(Q)
    q.qgemm_attention(Q, K_, V, O, scale=d["scale"])
    clean(f"attention {BH}x{Lq}x{Lk}")
    close(f"attention {BH}x{Lq}x{Lk}", O,
          oracle.attention(d["q"].numpy(), d["k"].numpy(), d["v"].numpy(), d["scale"]))
# decode GEMV with two activation halves and a ragged row block
gv = synth.w8_inputs(9, 1000, 512, seed=33)
W = q.qgemm_create_tensor(q.INT8, gv["w"].to(dev), gv["sw"].to(dev))
Y = torch.empty(9, 1000, dtype=torch.float16, device=dev)
q.qgemm_w8_gemv(gv["x"].to(dev), W, Y)
clean("gemv M=9")
close("gemv M=9", Y, oracle.w8_gemv(gv["x"].numpy(), gv["w"].numpy(), gv["sw"].numpy()))
print("DEBUG-BUILD-OK")
"""


def test_debug_build_every_route_clean():
    env = dict(os.environ, QGEMM_DEBUG="1", QG_ROOT=ROOT)
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, cwd=ROOT, capture_output=True,
                       text=True, timeout=1200)
    assert r.returncode == 0 and "DEBUG-BUILD-OK" in r.stdout, (r.stdout[-4000:] +
                                                               r.stderr[-4000:])
