"""Seeded synthetic inputs for the five workloads, on the CPU.

This module only draws random numbers and encodes them into the library's input formats.  It
holds none of the product's arithmetic (no decode, no product, no accumulation); the tests, the
benchmark and the smoke check feed the same bytes to both the CUDA path and the CPU oracle.

Workloads (all operands row-major, K contiguous, one UE8M0 scale per 32 elements along K):

* ``mxfp8_small``   -- MXFP8 M=128 N=256 K=128, source values N(0,1).
* ``f16_4096``      -- fp16 GEMM M=N=K=4096, A [M,K] and B [K,N] drawn N(0,1)/sqrt(K).
* ``mxfp8_8192``    -- MXFP8 M=N=K=8192; each row of A and of B gets variance 10^U(-2,2).
* ``w4a16_prefill`` -- fp16 A [4096,4096] N(0,1); int4 W [14336,4096] from N(0, 0.02^2).
* ``w8_decode``     -- fp16 X [M,8192] N(0,1), M in {1,8,16}; int8 W [28672,8192] from N(0, 0.02^2).
* ``mxfp4_8192``    -- MXFP4 M=N=K=8192; each row of A and of B gets variance 10^U(-2,2).
* ``w4a16_f16s_prefill`` -- as ``w4a16_prefill`` with fp16 block scales s = fp16(amax / 7).
* ``attn_prefill``  -- fused attention: Q, K, V fp16 [32 heads, 4096, 128] N(0,1), scale
  1/sqrt(128) (a bidirectional prefill of one sequence).

Encoding recipes (the pages only say "power-of-two block scales, 32 elements per block"; the
per-format details below are the workload definitions):

* MXFP8: per block X = floor(log2(amax)) - 8 (clamped to [-127, 127]), scale byte X + 127,
  element = E4M3(round-to-nearest-even(v / 2^X)) with saturation to +-448.  An all-zero block
  gets scale byte 127 and zero data.
* intN (N = 4 or 8, qmax = 7 or 127): scale s = 2^ceil(log2(amax / qmax)), byte log2(s) + 127,
  q = round-half-even(w / s) clamped to [-qmax-1, qmax].  int4 is packed two per byte, the even
  k in the low nibble ("TensorOps: quantized matmul ...", section "VALIDATED ON M4 MAX", fact 5).

* MXFP4: per block X = floor(log2(amax)) - 2 (E2M1's largest exponent is 2), scale byte X + 127,
  element = the nearest E2M1 value to v / 2^X (ties to the even code, i.e. mantissa bit 0),
  saturated to +-6; two per byte, even k in the low nibble (the int4 rule).

The E4M3 rounding is done by PyTorch's float8_e4m3fn cast (round-to-nearest-even) after the
saturating clamp; exponents come from ``torch.frexp`` so no ``log2`` rounding is involved.
"""
from __future__ import annotations

import math

import torch

BLOCK = 32
E4M3_MAX = 448.0


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal(shape, g: torch.Generator, std: float = 1.0) -> torch.Tensor:
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x


def _block_amax(x: torch.Tensor) -> torch.Tensor:
    rows, k = x.shape
    if k % BLOCK:
        raise ValueError("K must be a multiple of 32")
    return x.abs().reshape(rows, k // BLOCK, BLOCK).amax(dim=2)


def quantize_mxfp8(x: torch.Tensor):
    """fp32 [rows, K] -> (E4M3 bytes uint8 [rows, K], UE8M0 bytes uint8 [rows, K/32])."""
    x = x.to(torch.float32)
    rows, k = x.shape
    amax = _block_amax(x)
    _, e = torch.frexp(amax)                       # amax = f * 2^e, f in [0.5, 1)
    X = (e - 1 - 8).to(torch.int32)                # floor(log2(amax)) - 8
    X = torch.where(amax > 0, X, torch.zeros_like(X)).clamp(-127, 127)
    scale_bytes = (X + 127).to(torch.uint8)
    xs = x.reshape(rows, k // BLOCK, BLOCK)
    scaled = torch.ldexp(xs.to(torch.float64), (-X).to(torch.float64).unsqueeze(2))
    scaled = scaled.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float32)
    q = scaled.to(torch.float8_e4m3fn).view(torch.uint8).reshape(rows, k)
    return q.contiguous(), scale_bytes.contiguous()


E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)   # codes 0..7; 8..15 negative


def e2m1_round(y: torch.Tensor) -> torch.Tensor:
    """Codes 0..7 of the nearest E2M1 magnitude to |y| (fp64 y), ties to the even code, values
    above 6 saturated.  The spacing is 0.5 below 2, 1 in [2, 4) and 2 in [4, 6]; within each range
    an even multiple of the spacing is an even code, so half-to-even rounding of y / spacing is
    the tie rule."""
    y = y.abs().clamp(max=6.0)
    lo = torch.round(y / 0.5) * 0.5
    mid = torch.round(y)
    hi = torch.round(y / 2.0) * 2.0
    v = torch.where(y < 2.0, lo, torch.where(y < 4.0, mid, hi))
    grid = torch.tensor(E2M1_MAGNITUDES, dtype=torch.float64)
    return torch.searchsorted(grid, v.contiguous()).to(torch.uint8)


def quantize_mxfp4(x: torch.Tensor):
    """fp32 [rows, K] -> (packed E2M1 bytes uint8 [rows, K/2], UE8M0 bytes uint8 [rows, K/32])."""
    x = x.to(torch.float64)
    rows, k = x.shape
    amax = _block_amax(x)
    _, e = torch.frexp(amax)                       # amax = f * 2^e, f in [0.5, 1)
    X = (e - 1 - 2).to(torch.int32)                # floor(log2(amax)) - 2
    X = torch.where(amax > 0, X, torch.zeros_like(X)).clamp(-127, 127)
    scale_bytes = (X + 127).to(torch.uint8)
    xs = x.reshape(rows, k // BLOCK, BLOCK)
    scaled = torch.ldexp(xs, (-X).to(torch.float64).unsqueeze(2)).reshape(rows, k)
    code = e2m1_round(scaled) | (torch.signbit(scaled).to(torch.uint8) << 3)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).to(torch.uint8)
    return packed.contiguous(), scale_bytes.contiguous()


def quantize_int_blocks(w: torch.Tensor, qmax: int):
    """fp32 [rows, K] -> (int8 values [rows, K] in [-qmax-1, qmax], UE8M0 bytes [rows, K/32])."""
    w = w.to(torch.float64)
    rows, k = w.shape
    amax = _block_amax(w)
    y = amax / qmax
    f, e = torch.frexp(y)                          # y = f * 2^e
    c = torch.where(f == 0.5, e - 1, e)            # ceil(log2(y)); exact powers of two stay
    c = torch.where(amax > 0, c, torch.zeros_like(c)).clamp(-127, 127)
    scale_bytes = (c + 127).to(torch.uint8)
    ws = w.reshape(rows, k // BLOCK, BLOCK)
    q = torch.round(torch.ldexp(ws, (-c).to(torch.float64).unsqueeze(2)))  # half to even
    q = q.clamp(-qmax - 1, qmax).to(torch.int8).reshape(rows, k)
    return q.contiguous(), scale_bytes.contiguous()


def quantize_int4_f16_scales(w: torch.Tensor):
    """fp32 [rows, K] -> (int8 values [rows, K] in [-8, 7], fp16 scales [rows, K/32]).

    The custom (non-MX) format: each block's scale is the fp16 value nearest to amax / 7 (1.0 for
    an all-zero block), not a power of two; q = round_half_even(w / s) clamped to [-8, 7]."""
    w = w.to(torch.float64)
    rows, k = w.shape
    amax = _block_amax(w)
    s16 = torch.where(amax > 0, amax / 7.0, torch.ones_like(amax)).to(torch.float16)
    s64 = s16.to(torch.float64)
    ws = w.reshape(rows, k // BLOCK, BLOCK)
    q = torch.round(ws / s64.unsqueeze(2)).clamp(-8, 7).to(torch.int8).reshape(rows, k)
    return q.contiguous(), s16.contiguous()


def pack_int4(q: torch.Tensor) -> torch.Tensor:
    """int8 values in [-8, 7], [rows, K] -> packed uint8 [rows, K/2], even k in the low nibble."""
    rows, k = q.shape
    if k % 2:
        raise ValueError("K must be even for int4")
    u = (q.to(torch.int16) & 0xF).to(torch.uint8).reshape(rows, k // 2, 2)
    return (u[:, :, 0] | (u[:, :, 1] << 4)).contiguous()


def log_uniform_row_std(rows: int, g: torch.Generator, lo_exp=-2.0, hi_exp=2.0) -> torch.Tensor:
    """Per-row standard deviation sqrt(10^U(lo, hi))."""
    u = torch.rand(rows, generator=g, dtype=torch.float64) * (hi_exp - lo_exp) + lo_exp
    return torch.sqrt(torch.pow(10.0, u)).to(torch.float32)


# ------------------------------------------------------------------------------ workloads
WORKLOADS = ("mxfp8_small", "f16_4096", "mxfp8_8192", "w4a16_prefill", "w8_decode", "mxfp4_8192",
             "w4a16_f16s_prefill", "attn_prefill")


def mxfp8_inputs(M: int, N: int, K: int, seed: int, row_variance: bool = False):
    """MXFP8 operands: A [M,K], B [N,K] (E4M3 bytes) with UE8M0 scales [rows, K/32]."""
    g = generator(seed)
    if row_variance:
        sa = log_uniform_row_std(M, g)
        sb = log_uniform_row_std(N, g)
        a = normal((M, K), g) * sa[:, None]
        b = normal((N, K), g) * sb[:, None]
    else:
        a = normal((M, K), g)
        b = normal((N, K), g)
    qa, sa_b = quantize_mxfp8(a)
    qb, sb_b = quantize_mxfp8(b)
    return {"a": qa, "sa": sa_b, "b": qb, "sb": sb_b, "M": M, "N": N, "K": K}


def mxfp4_inputs(M: int, N: int, K: int, seed: int, row_variance: bool = False):
    """MXFP4 operands: A [M,K/2], B [N,K/2] (packed E2M1 bytes) with UE8M0 scales [rows, K/32]."""
    g = generator(seed)
    if row_variance:
        sa = log_uniform_row_std(M, g)
        sb = log_uniform_row_std(N, g)
        a = normal((M, K), g) * sa[:, None]
        b = normal((N, K), g) * sb[:, None]
    else:
        a = normal((M, K), g)
        b = normal((N, K), g)
    qa, sa_b = quantize_mxfp4(a)
    qb, sb_b = quantize_mxfp4(b)
    return {"a": qa, "sa": sa_b, "b": qb, "sb": sb_b, "M": M, "N": N, "K": K}


def f16_inputs(M: int, N: int, K: int, seed: int):
    g = generator(seed)
    s = 1.0 / math.sqrt(K)
    a = (normal((M, K), g) * s).to(torch.float16)
    b = (normal((K, N), g) * s).to(torch.float16)
    return {"a": a.contiguous(), "b": b.contiguous(), "M": M, "N": N, "K": K}


def w4a16_inputs(M: int, N: int, K: int, seed: int, w_std: float = 0.02):
    g = generator(seed)
    a = normal((M, K), g).to(torch.float16)
    w = normal((N, K), g, std=w_std)
    q, s = quantize_int_blocks(w, 7)
    return {"a": a.contiguous(), "w": pack_int4(q), "w_values": q, "sw": s,
            "M": M, "N": N, "K": K}


def w4a16_f16s_inputs(M: int, N: int, K: int, seed: int, w_std: float = 0.02):
    """fp16 A [M,K] N(0,1); int4 W [N,K] (packed) with fp16 block scales [N,K/32]."""
    g = generator(seed)
    a = normal((M, K), g).to(torch.float16)
    w = normal((N, K), g, std=w_std)
    q, s = quantize_int4_f16_scales(w)
    return {"a": a.contiguous(), "w": pack_int4(q), "w_values": q, "sw": s,
            "M": M, "N": N, "K": K}


W4_SCALE_KINDS = 9


def w4a16_scale_extremes_inputs(M: int, N: int, K: int, seed: int):
    """int4 weights whose UE8M0 scale bytes span the whole byte range, within rows and across
    them, with activations shaped so that the outputs stay well inside the fp16 range.

    Activations: N(0, 1) times 2^8 on even 32-blocks of k and times 2^-12 on odd ones, so a
    block with a small scale byte is placed on an even block and one with a large byte on an
    odd block.  Weight row n is of kind n % 9 (``kind`` in the result):
      0  every block live, bytes in 103..117 (even blocks) / 118..139 (odd blocks);
      1  kind 0 with four blocks emptied (all q = 0) under bytes from {0, 1, 60, 102, 140, 180, 254};
      2  live even blocks under bytes 102, 60, 1 and 0 only (every other block emptied);
      3  kind 0 plus one or two live odd blocks under bytes from {140, 143, 146};
      4  kind 0 plus live {0, 1, 60, 102} (even), one live 140 or 146 (odd), empty 180 and 254;
      5  kind 0 with one live block under byte 255 (NaN);
      6  kind 0 with one empty block under byte 255;
      7  kind 0 with one live odd block under byte 180 or 254 (overflows fp16);
      8  every block live under byte 102.
    Kinds 2, 3, 4, 7 and 8 hold nonzero weights in blocks whose byte is outside 103..139 and
    not 255."""
    g = generator(seed)
    nblk = K // BLOCK
    if nblk < 8:
        raise ValueError("K must be at least 256")
    even = torch.arange(nblk) % 2 == 0
    amp = torch.where(even, 2.0 ** 8, 2.0 ** -12).repeat_interleave(BLOCK)
    a = (normal((M, K), g) * amp).to(torch.float16)
    q = torch.randint(-8, 8, (N, K), generator=g, dtype=torch.int8)
    q[q == 0] = 1                              # every block of a live row holds nonzero weights
    sw = torch.empty(N, nblk, dtype=torch.uint8)
    sw[:, even] = torch.randint(103, 118, (N, int(even.sum())), generator=g, dtype=torch.uint8)
    sw[:, ~even] = torch.randint(118, 140, (N, int((~even).sum())), generator=g, dtype=torch.uint8)
    ev_idx = torch.nonzero(even).flatten()
    od_idx = torch.nonzero(~even).flatten()

    def pick(idx, n_pick):
        return idx[torch.randperm(idx.numel(), generator=g)[:n_pick]]

    def choice(vals, n_pick):
        v = torch.tensor(vals, dtype=torch.uint8)
        return v[torch.randint(0, len(vals), (n_pick,), generator=g)]

    def empty_block(n, b):
        q[n, b * BLOCK:(b + 1) * BLOCK] = 0

    kind = torch.arange(N) % W4_SCALE_KINDS
    for n in range(N):
        k_ = int(kind[n])
        if k_ == 1:
            bs = pick(torch.arange(nblk), 4)
            sw[n, bs] = choice([0, 1, 60, 102, 140, 180, 254], 4)
            for b in bs.tolist():
                empty_block(n, b)
        elif k_ == 2:
            bs = pick(ev_idx, 4)
            sw[n, bs] = torch.tensor([102, 60, 1, 0], dtype=torch.uint8)
            keep = set(bs.tolist())
            for b in range(nblk):
                if b not in keep:
                    empty_block(n, b)
        elif k_ == 3:
            bs = pick(od_idx, 1 + int(torch.randint(0, 2, (1,), generator=g)))
            sw[n, bs] = choice([140, 143, 146], bs.numel())
        elif k_ == 4:
            be = pick(ev_idx, 4)
            sw[n, be] = torch.tensor([0, 1, 60, 102], dtype=torch.uint8)
            bo = pick(od_idx, 3)
            sw[n, bo] = torch.tensor([int(choice([140, 146], 1)), 180, 254], dtype=torch.uint8)
            empty_block(n, int(bo[1]))
            empty_block(n, int(bo[2]))
        elif k_ == 5:
            sw[n, int(pick(torch.arange(nblk), 1))] = 255
        elif k_ == 6:
            b = int(pick(torch.arange(nblk), 1))
            sw[n, b] = 255
            empty_block(n, b)
        elif k_ == 7:
            sw[n, int(pick(od_idx, 1))] = 180 if (n // W4_SCALE_KINDS) % 2 == 0 else 254
        elif k_ == 8:
            sw[n, :] = 102
    return {"a": a.contiguous(), "w": pack_int4(q), "w_values": q, "sw": sw.contiguous(),
            "kind": kind, "M": M, "N": N, "K": K}


def attention_inputs(BH: int, Lq: int, Lk: int, d: int, seed: int, q_std: float = 1.0):
    """fp16 Q [BH, Lq, d], K and V [BH, Lk, d] from N(0, 1) (Q times q_std: a larger q_std makes
    the softmax rows peakier); scale 1/sqrt(d)."""
    g = generator(seed)
    q = (normal((BH, Lq, d), g) * q_std).to(torch.float16)
    k = normal((BH, Lk, d), g).to(torch.float16)
    v = normal((BH, Lk, d), g).to(torch.float16)
    return {"q": q.contiguous(), "k": k.contiguous(), "v": v.contiguous(), "scale": d ** -0.5,
            "BH": BH, "Lq": Lq, "Lk": Lk, "d": d}


def w8_inputs(M: int, N: int, K: int, seed: int, w_std: float = 0.02):
    g = generator(seed)
    x = normal((M, K), g).to(torch.float16)
    w = normal((N, K), g, std=w_std)
    q, s = quantize_int_blocks(w, 127)
    return {"x": x.contiguous(), "w": q.view(torch.uint8).contiguous(), "sw": s,
            "M": M, "N": N, "K": K}


def workload(name: str, M: int | None = None):
    """Full-size inputs of a named workload (seed = its position in ``WORKLOADS``)."""
    seed = WORKLOADS.index(name)
    if name == "mxfp8_small":
        return mxfp8_inputs(128, 256, 128, seed)
    if name == "f16_4096":
        return f16_inputs(4096, 4096, 4096, seed)
    if name == "mxfp8_8192":
        return mxfp8_inputs(8192, 8192, 8192, seed, row_variance=True)
    if name == "w4a16_prefill":
        return w4a16_inputs(4096, 14336, 4096, seed)
    if name == "w8_decode":
        return w8_inputs(16 if M is None else M, 28672, 8192, seed)
    if name == "mxfp4_8192":
        return mxfp4_inputs(8192, 8192, 8192, seed, row_variance=True)
    if name == "w4a16_f16s_prefill":
        return w4a16_f16s_inputs(4096, 14336, 4096, seed)
    if name == "attn_prefill":
        return attention_inputs(32, 4096, 4096, 128, seed)
    raise KeyError(name)
