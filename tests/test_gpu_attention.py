"""GPU parity of the fused attention kernel (qgemm_attention_f16) against the oracle's fp64
softmax attention, through the C ABI.

Tolerance (element-wise): |O_gpu - O| <= 2e-3 * D + 2^-24 with D = sum_j p_j |v_j| / sum_j p_j,
the magnitude the weighted average is formed from.
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


def _check(got, res, orc, what):
    code = q.qgemm_poll_device_error()
    assert code == 0, f"{what}: a device wait timed out (error word {code:#x})"
    g = got.float().cpu().numpy().reshape(res.C.shape)
    ok, worst, info = orc.within_tolerance(g, res, REL)
    assert ok, f"{what}: {info}"
    return worst


def _run(d, dev, layout="bhld"):
    Q, K, V = d["q"].to(dev), d["k"].to(dev), d["v"].to(dev)
    O = torch.full_like(Q, float("nan"))
    q.qgemm_attention(Q, K, V, O, scale=d["scale"])
    return O


@pytest.mark.parametrize("BH,Lq,Lk,q_std", [(2, 128, 128, 1.0), (3, 200, 300, 1.0),
                                            (1, 1, 1, 1.0), (2, 257, 1000, 2.0),
                                            (4, 512, 640, 4.0), (1, 384, 2048, 8.0)])
def test_attention_matches_oracle(dev, orc, BH, Lq, Lk, q_std):
    d = synth.attention_inputs(BH, Lq, Lk, 128, seed=BH + Lq + Lk, q_std=q_std)
    O = _run(d, dev)
    res = orc.attention(d["q"].numpy(), d["k"].numpy(), d["v"].numpy(), d["scale"])
    _check(O, res, orc, f"attention {BH}x{Lq}x{Lk} q_std={q_std}")


def test_attention_rising_maximum_rescales(dev, orc):
    """Keys whose norm grows along the sequence: every key tile raises the row maximum by more
    than 2^8, so the output accumulator is rescaled on every tile."""
    BH, Lq, Lk = 2, 256, 1024
    d = synth.attention_inputs(BH, Lq, Lk, 128, seed=71)
    growth = torch.linspace(0.2, 3.0, Lk).reshape(1, Lk, 1)
    d["k"] = (d["k"].float() * growth).to(torch.float16)
    d["q"] = (d["q"].float() * 2.0).to(torch.float16)
    O = _run(d, dev)
    res = orc.attention(d["q"].numpy(), d["k"].numpy(), d["v"].numpy(), d["scale"])
    _check(O, res, orc, "attention rising maximum")


def test_attention_single_key_is_exact(dev):
    """One key: every softmax weight is exactly 1 and O is that value row, bit for bit."""
    d = synth.attention_inputs(3, 130, 1, 128, seed=72)
    O = _run(d, dev)
    torch.cuda.synchronize()
    assert torch.equal(O.cpu(), d["v"].expand(3, 130, 128))


def test_attention_interleaved_heads_layout(dev, orc):
    """[L, heads, d] buffers (row stride = heads * d, head stride = d) for Q, K, V and O."""
    H, Lq, Lk = 4, 192, 320
    d = synth.attention_inputs(H, Lq, Lk, 128, seed=73, q_std=2.0)
    Qi = d["q"].transpose(0, 1).contiguous().to(dev)     # [Lq, H, d]
    Ki = d["k"].transpose(0, 1).contiguous().to(dev)
    Vi = d["v"].transpose(0, 1).contiguous().to(dev)
    Oi = torch.full((Lq, H, 128), float("nan"), dtype=torch.float16, device=dev)
    q.qgemm_attention(Qi.transpose(0, 1), Ki.transpose(0, 1), Vi.transpose(0, 1),
                      Oi.transpose(0, 1), scale=d["scale"])
    res = orc.attention(d["q"].numpy(), d["k"].numpy(), d["v"].numpy(), d["scale"])
    _check(Oi.transpose(0, 1), res, orc, "attention interleaved heads")


def _parts(units, nkv, sms, min_range=4):
    """The kernel's work split, restated on the host for the tests' assertions: whole waves of
    units data-parallel while at least two waves remain, then the key tiles of the units left
    in equal contiguous ranges, one per CTA.  Returns (CTAs, per CTA the list of (unit, first
    key tile, key tiles, kind)) with kind 'whole', 'tail' (range starts inside the unit) or
    'head' (range ends inside it)."""
    G = max(1, min(sms, units * nkv // min_range))
    D = units // G - 1 if units // G >= 2 else 0
    u0, T = D * G, (units - D * G) * nkv
    start = lambda c: c * (T // G) + min(c, T % G)
    out = []
    for c in range(G):
        parts = [(w * G + c, 0, nkv, "whole") for w in range(D)]
        cur, end = start(c), start(c + 1)
        while cur < end:
            u, kv0 = divmod(cur, nkv)
            n = min(end, (u + 1) * nkv) - cur
            kind = "tail" if kv0 > 0 else ("head" if cur + n < (u + 1) * nkv else "whole")
            parts.append((u0 + u, kv0, n, kind))
            cur += n
        out.append(parts)
    return G, out


def _check_split_case(dev, orc, BH, Lq, Lk, seed, what):
    d = synth.attention_inputs(BH, Lq, Lk, 128, seed=seed, q_std=2.0)
    O = _run(d, dev)
    res = orc.attention(d["q"].numpy(), d["k"].numpy(), d["v"].numpy(), d["scale"])
    _check(O, res, orc, f"{what} {BH}x{Lq}x{Lk}")
    O2 = _run(d, dev)
    assert torch.equal(O2.view(torch.int16), O.view(torch.int16))     # repeatable bit for bit


def test_attention_waves_then_ranges(dev, orc):
    """More than two waves of units (head, 256 query rows): whole waves run data-parallel, and
    the units left are shared out in key-tile ranges whose boundaries cut units into a tail
    (its CTA's first part) and a head (another CTA's last part), merged in the head's output.
    Lk = 600 puts the ragged key tile in the tails."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    BH, Lq, Lk = (2 * sms + 7) // 4 + 1, 1024, 600
    units, nkv = BH * 4, (Lk + 127) // 128
    G, parts = _parts(units, nkv, sms)
    assert units // G >= 2                                          # a data-parallel wave
    kinds = [k for p in parts for (_, _, _, k) in p]
    assert "tail" in kinds and "head" in kinds
    _check_split_case(dev, orc, BH, Lq, Lk, 74, "attention waves + ranges")


def test_attention_ranges_only(dev, orc):
    """Between one and two waves of units: no data-parallel wave, every CTA's work is a range,
    some CTAs both finish a unit's tail first and start another unit's head last."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    BH, Lq, Lk = (sms + 4) // 4 + 1, 1024, 1000
    units, nkv = BH * 4, (Lk + 127) // 128
    G, parts = _parts(units, nkv, sms)
    assert G == sms and units // G == 1
    assert any(p[0][3] == "tail" and p[-1][3] == "head" for p in parts)
    _check_split_case(dev, orc, BH, Lq, Lk, 75, "attention ranges")


@pytest.mark.parametrize("BH,Lq,Lk", [(1, 256, 8192), (1, 100, 4096), (2, 300, 2000),
                                      (1, 256, 65536), (1, 1, 4096), (3, 1, 2048)])
def test_attention_unit_over_many_ctas(dev, orc, BH, Lq, Lk):
    """Fewer units than SMs: a unit's key tiles spread over several CTAs, whose head part merges
    several tails (127 of them for one unit over 65536 keys); Lq = 100, 300 and 1 leave rows of a
    merged unit past Lq (computed, not stored)."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    units, nkv = BH * ((Lq + 255) // 256), (Lk + 127) // 128
    G, parts = _parts(units, nkv, sms)
    tails = max(sum(1 for p in parts for (u, _, _, k) in p if k == "tail" and u == uu)
                for uu in range(units))
    assert tails >= 2
    _check_split_case(dev, orc, BH, Lq, Lk, 76 + Lq, "attention unit over many CTAs")


def test_attention_errors(dev):
    x = torch.zeros(1, 16, 64, dtype=torch.float16, device=dev)
    with pytest.raises(q.QGemmError) as ei:
        q.qgemm_attention(x, x, x, x.clone())
    assert ei.value.name == "QGEMM_ERR_UNSUPPORTED_SHAPE"          # d != 128
    y = torch.zeros(1, 16, 128, dtype=torch.float16, device=dev)
    k0 = torch.zeros(1, 0, 128, dtype=torch.float16, device=dev)
    with pytest.raises(q.QGemmError) as ei:
        q.qgemm_attention(y, k0, k0, y.clone())
    assert ei.value.name == "QGEMM_ERR_UNSUPPORTED_SHAPE"          # Lk = 0
    with pytest.raises(q.QGemmError) as ei:
        q.qgemm_attention(y, y, y, y.clone(), scale=-1.0)
    assert ei.value.name == "QGEMM_ERR_INVALID_ARG"
    big = torch.zeros(1, 16, 136, dtype=torch.float16, device=dev)
    with pytest.raises(q.QGemmError) as ei:
        q.qgemm_attention(big[:, :, 4:132], y, y, y.clone())           # base not 16-byte aligned
    assert ei.value.name == "QGEMM_ERR_MISALIGNED"


def test_attention_full_size_sampled(dev, orc):
    """32 heads x 4096 x 4096 x 128 (the prefill workload), oracle on sampled rows."""
    d = synth.workload("attn_prefill")
    O = _run(d, dev)
    rng = np.random.default_rng(4)
    heads = np.concatenate([[0, 31], rng.integers(0, 32, 30)])
    rows = np.concatenate([[0, 4095], rng.integers(0, 4096, 30)])
    res = orc.attention(d["q"].numpy(), d["k"].numpy(), d["v"].numpy(), d["scale"],
                        heads=heads, qrows=rows)
    got = O[torch.from_numpy(heads).to(dev), torch.from_numpy(rows).to(dev)]
    _check(got, res, orc, "attention 32x4096x4096 sampled")
    O2 = _run(d, dev)
    assert torch.equal(O2.view(torch.int16), O.view(torch.int16))     # repeatable bit for bit
