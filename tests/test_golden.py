"""The oracle against the golden fixtures under tests/golden/ (no GPU needed).

Each fixture holds values worked by hand from the pages' statement of the formats, or values the
pages print; its header names the page and section.  The fixtures are read here as text; nothing in
them comes from the oracle or from the CUDA path.
"""
import os
from fractions import Fraction

import numpy as np
import torch

from block_scaled_quantized_tcgen05_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                yield line.strip()


def parse_entries(spec: str, K: int) -> np.ndarray:
    """'0-15:38,32:b8' -> K bytes, the listed codes at the listed k and 0x00 elsewhere."""
    v = np.zeros(K, np.uint8)
    for part in spec.split(","):
        ks, code = part.split(":")
        lo, _, hi = ks.partition("-")
        v[int(lo):int(hi or lo) + 1] = int(code, 16)
    return v


def mxfp8_cases(K: int = 64):
    """(name, A [1,K], SA [1,K/32], B [1,K], SB [1,K/32], C, D, fp16 bits or None for NaN)."""
    for line in _lines("mxfp8_hand_worked.txt"):
        name, a, sa, b, sb, c, d, bits = (x.strip() for x in line.split("|"))
        A = parse_entries(a, K)[None, :]
        B = parse_entries(b, K)[None, :]
        SA = np.array([[int(x) for x in sa.split(",")]], np.uint8)
        SB = np.array([[int(x) for x in sb.split(",")]], np.uint8)
        C = None if c == "nan" else Fraction(c)
        D = None if d == "nan" else Fraction(d)
        yield name, A, SA, B, SB, C, D, None if bits == "nan" else int(bits, 16)


def test_int4_packing_follows_the_page(orc):
    """Every hand-packed byte decodes to its two values (even k in the low nibble), and the input
    generators' packer produces the same byte."""
    rows = [line.split() for line in _lines("int4_packing.txt")]
    assert len(rows) >= 8
    for v0, v1, byte in rows:
        b = np.array([int(byte, 16)], np.uint8)
        assert orc.int4_get(b, 0) == int(v0) and orc.int4_get(b, 1) == int(v1)
        packed = synth.pack_int4(torch.tensor([[int(v0), int(v1)]], dtype=torch.int8))
        assert int(packed.numpy()[0, 0]) == int(byte, 16)


def test_mxfp8_hand_worked_products(orc):
    """Exact product, magnitude sum and fp16 bits of every hand-worked MXFP8 case."""
    n = 0
    for name, A, SA, B, SB, C, D, bits in mxfp8_cases():
        res = orc.mxfp8(A, SA, B, SB)
        if bits is None:
            assert np.isnan(res.C[0, 0]) and np.isnan(res.f16[0, 0]), name
        else:
            assert Fraction(float(res.C[0, 0])) == C, name
            assert Fraction(float(res.D[0, 0])) == D, name
            assert int(res.f16_bits[0, 0]) == bits, name
        n += 1
    assert n >= 15


def test_validation_table_cosine(orc):
    """The pages print cos-sim 1.000000 against a torch reference for each variant; the oracle's
    products on the same operands agree with a library matmul to that printed precision."""
    rows = [[x.strip() for x in line.split("|")] for line in _lines("validation_cos_sim.txt")]
    assert [r[0] for r in rows] == ["M0", "M1a", "M1b", "M2"]
    for kernel, _, shape, printed in rows:
        M, K, N = (int(x) for x in shape.split())
        res, ref = validation_case(orc, kernel, M, K, N)
        assert f"{orc.cosine(res.C, ref):.6f}" == printed, kernel


def validation_case(orc, kernel, M, K, N, seed=7):
    """Oracle result and the torch fp32 reference for one row of the validation table, on seeded
    inputs of the pages' kind (activations N(0,1) in fp16, weights N(0, 0.02))."""
    g = synth.generator(seed)
    x = synth.normal((M, K), g).to(torch.float16)
    w = synth.normal((N, K), g, std=0.02)
    if kernel == "M0":
        b = w.to(torch.float16).t().contiguous()                 # [K, N] row-major
        res = orc.gemm_f16(x.numpy(), b.numpy())
        wd = b.t().float()
    elif kernel == "M1a":
        d = validation_int_weights(w, 127)
        res = orc.w8_gemv(x.numpy(), d["q"].view(torch.uint8).numpy(), d["s"].numpy())
        wd = d["deq"]
    elif kernel == "M1b":
        d = validation_int_weights(w, 7)
        packed = synth.pack_int4(d["q"])
        res = orc.w4a16(x.numpy(), packed.numpy(), d["s"].numpy())
        wd = d["deq"]
    else:
        d = synth.w4a16_f16s_inputs(M, N, K, seed)
        x = d["a"]
        res = orc.w4a16_f16s(x.numpy(), d["w"].numpy(), d["sw"].numpy())
        wd = torch.from_numpy(orc.dequant_int4_f16s(d["w"].numpy(), d["sw"].numpy()))
    ref = (x.float() @ wd.float().t()).numpy()
    return res, ref


def validation_int_weights(w: torch.Tensor, qmax: int):
    """Uniform (per-tensor) power-of-two scale: every block shares one scale byte."""
    amax = float(w.abs().max())
    e = int(np.ceil(np.log2(amax / qmax)))
    s = 2.0 ** e
    q = torch.clamp(torch.round(w / s), -qmax - 1, qmax).to(torch.int8)
    sc = torch.full((w.shape[0], w.shape[1] // 32), 127 + e, dtype=torch.uint8)
    return {"q": q, "s": sc, "deq": q.float() * s}
