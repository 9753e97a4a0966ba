"""The seeded input encoders follow the workload recipes (checked element by element against a
plain-Python restatement on small blocks, and by properties on large ones)."""
import math

import numpy as np
import torch

from block_scaled_quantized_tcgen05_gb300 import synth


def _nearest_e4m3_code(v: float, table: np.ndarray) -> int:
    """Round-to-nearest-even onto the finite E4M3 grid, saturating at +-448."""
    v = max(-448.0, min(448.0, v))
    best = None
    for code in range(256):
        t = table[code]
        if not np.isfinite(t):
            continue
        d = abs(t - v)
        key = (d, code & 1)                      # ties -> even mantissa (code LSB 0)
        if best is None or key < best[0] or (key == best[0] and code < best[1]):
            best = (key, code)
    code = best[1]
    if v == 0.0:
        return 0x80 if math.copysign(1.0, v) < 0 else 0x00
    return code


def test_mxfp8_quantizer_matches_plain_restatement(orc):
    table = orc.e4m3_table()
    g = synth.generator(123)
    x = synth.normal((6, 64), g) * torch.tensor([[1e-3], [1.0], [300.0], [1e-30], [7.0], [0.0]])
    x[4, 5] = -x[4, :32].abs().max() * 1.0001                     # negative amax
    q, s = synth.quantize_mxfp8(x)
    for r in range(x.shape[0]):
        for b in range(2):
            blk = x[r, 32 * b:32 * b + 32].double().numpy()
            amax = float(np.abs(blk).max())
            X = 0 if amax == 0 else max(-127, min(127, math.floor(math.log2(amax)) - 8))
            if amax > 0:   # math.log2 can round; fix up with exact comparisons
                while 2.0 ** (X + 8) > amax:
                    X -= 1
                while 2.0 ** (X + 9) <= amax:
                    X += 1
                X = max(-127, min(127, X))
            assert int(s[r, b]) == X + 127
            for j in range(32):
                want = _nearest_e4m3_code(blk[j] / 2.0 ** X, table)
                got = int(q[r, 32 * b + j])
                assert table[got] == table[want], (r, b, j, blk[j], got, want)


def test_mxfp8_quantizer_properties(orc):
    table = orc.e4m3_table()
    d = synth.mxfp8_inputs(64, 32, 256, seed=7, row_variance=True)
    q = d["a"].numpy()
    s = d["sa"].numpy().astype(np.int64)
    vals = table[q]
    assert np.isfinite(vals).all()
    blk_max = np.abs(vals).reshape(64, 8, 32).max(axis=2)
    assert np.all((blk_max >= 256) & (blk_max <= 448))          # amax lands in [256, 448]
    assert np.all((s >= 1) & (s <= 254))


def test_int_quantizers_match_plain_restatement():
    g = synth.generator(9)
    w = synth.normal((4, 96), g, std=0.02)
    w[2, :32] = 0.0
    w[3, 40] = 0.07                                             # amax/7 = 0.01 exactly? no: pow2 check
    for qmax in (7, 127):
        q, s = synth.quantize_int_blocks(w, qmax)
        for r in range(4):
            for b in range(3):
                blk = w[r, 32 * b:32 * b + 32].double().numpy()
                amax = float(np.abs(blk).max())
                if amax == 0:
                    c = 0
                else:
                    c = math.ceil(math.log2(amax / qmax))
                    while 2.0 ** (c - 1) >= amax / qmax:
                        c -= 1
                    while 2.0 ** c < amax / qmax:
                        c += 1
                assert int(s[r, b]) == c + 127
                want = np.clip(np.round(blk / 2.0 ** c), -qmax - 1, qmax)   # numpy: half to even
                assert np.array_equal(q[r, 32 * b:32 * b + 32].numpy(), want.astype(np.int8))


def test_workload_shapes_small():
    d = synth.workload("mxfp8_small")
    assert d["a"].shape == (128, 128) and d["b"].shape == (256, 128)
    assert d["sa"].shape == (128, 4) and d["sb"].shape == (256, 4)
    d2 = synth.workload("mxfp8_small")
    assert torch.equal(d["a"], d2["a"]) and torch.equal(d["sb"], d2["sb"])   # seeded


def _nearest_e2m1_code(y: float, table: np.ndarray) -> int:
    """Nearest E2M1 value to y over all 16 codes, saturating at +-6; ties go to the code whose
    mantissa bit (bit 0) is clear; the sign follows y."""
    y = max(-6.0, min(6.0, y))
    best = None
    for code in range(16):
        if (code >> 3) != (1 if math.copysign(1.0, y) < 0 else 0):
            continue
        key = (abs(float(table[code]) - y), code & 1)
        if best is None or key < best[0]:
            best = (key, code)
    return best[1]


def test_mxfp4_quantizer_matches_plain_restatement(orc):
    table = orc.e2m1_table()
    g = synth.generator(321)
    x = synth.normal((5, 64), g) * torch.tensor([[1e-3], [1.0], [50.0], [1e-30], [0.0]])
    x[1, 3] = -x[1, :32].abs().max() * 1.0001                     # negative amax
    x[2, 40:44] = torch.tensor([0.25, 0.75, 2.5, 5.0]) * 2.0 ** math.floor(
        math.log2(float(x[2, 32:].abs().max())) - 2)             # exact ties on the grid
    p, s = synth.quantize_mxfp4(x)
    assert p.shape == (5, 32) and s.shape == (5, 2)
    for r in range(x.shape[0]):
        for b in range(2):
            blk = x[r, 32 * b:32 * b + 32].double().numpy()
            amax = float(np.abs(blk).max())
            X = 0
            if amax > 0:
                X = math.floor(math.log2(amax)) - 2
                while 2.0 ** (X + 2) > amax:
                    X -= 1
                while 2.0 ** (X + 3) <= amax:
                    X += 1
                X = max(-127, min(127, X))
            assert int(s[r, b]) == X + 127
            for j in range(32):
                k = 32 * b + j
                byte = int(p[r, k // 2])
                got = (byte >> 4) if k % 2 else (byte & 15)
                want = _nearest_e2m1_code(blk[j] / 2.0 ** X, table)
                assert table[got] == table[want], (r, b, j, blk[j], got, want)


def test_mxfp4_quantizer_properties(orc):
    table = orc.e2m1_table()
    d = synth.mxfp4_inputs(64, 32, 256, seed=8, row_variance=True)
    p = d["a"].numpy()
    codes = np.stack([p & 15, p >> 4], axis=2).reshape(64, 256)
    vals = table[codes]
    blk_max = np.abs(vals).reshape(64, 8, 32).max(axis=2)
    assert np.all((blk_max >= 4) & (blk_max <= 6))               # amax lands in [4, 6]
    s = d["sa"].numpy().astype(np.int64)
    assert np.all((s >= 1) & (s <= 254))


def test_int4_f16_scale_encoder_matches_plain_restatement():
    g = synth.generator(10)
    w = synth.normal((3, 96), g, std=0.02)
    w[1, 32:64] = 0.0
    q, s = synth.quantize_int4_f16_scales(w)
    assert q.dtype == torch.int8 and s.dtype == torch.float16 and s.shape == (3, 3)
    for r in range(3):
        for b in range(3):
            blk = w[r, 32 * b:32 * b + 32].double().numpy()
            amax = float(np.abs(blk).max())
            want_s = np.float16(amax / 7.0) if amax > 0 else np.float16(1.0)
            assert s[r, b].item() == float(want_s)
            want_q = np.clip(np.round(blk / float(want_s)), -8, 7)       # half to even
            assert np.array_equal(q[r, 32 * b:32 * b + 32].numpy(), want_q.astype(np.int8))


def test_w4a16_scale_extremes_row_kinds():
    """The scale-extremes workload holds what its row kinds promise: live blocks (some nonzero
    weight) under bytes outside 103..139 exactly in kinds 2, 3, 4, 7 and 8; byte 255 in kinds 5
    and 6 (live in 5, emptied in 6); and bytes 0, 1, 60, 102, 140, 180, 254 all present."""
    N, K = 90, 1024
    d = synth.w4a16_scale_extremes_inputs(8, N, K, seed=3)
    qv = d["w_values"].numpy().reshape(N, K // 32, 32)
    sw = d["sw"].numpy().astype(np.int64)
    kind = d["kind"].numpy()
    live = (qv != 0).any(axis=2)
    outside = ((sw < 103) | (sw > 139)) & (sw != 255)
    has_live_outside = (live & outside).any(axis=1)
    assert np.array_equal(has_live_outside, np.isin(kind, [2, 3, 4, 7, 8]))
    nan_live = ((sw == 255) & live).any(axis=1)
    nan_dead = ((sw == 255) & ~live).any(axis=1)
    assert np.array_equal(nan_live, kind == 5) and np.array_equal(nan_dead, kind == 6)
    for byte in (0, 1, 60, 102, 140, 180, 254, 255):
        assert (sw == byte).any(), byte
    # packing agrees with the values (even k in the low nibble)
    p = d["w"].numpy()
    lo = (p & 15).astype(np.int8)
    hi = (p >> 4).astype(np.int8)
    unpacked = np.stack([np.where(lo > 7, lo - 16, lo), np.where(hi > 7, hi - 16, hi)],
                        axis=2).reshape(N, K)
    assert np.array_equal(unpacked, d["w_values"].numpy())
