"""Seeded synthetic inputs for the MXFP8 activation chain.

This module draws numbers and nothing else: it holds none of the quantizer's, the GEMMs' or
the RMSNorm's arithmetic, so both the GPU library's tests/bench and the CPU oracle can take
their inputs from it. It imports neither of them.

Generator: counter-based SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014). Element ``i`` of stream ``key`` is
``mix64(key + (i + 1) * 0x9E3779B97F4A7C15)``; uniforms take the top 53 bits; normals use the
Box-Muller transform (1958) in fp64, then round fp64 -> fp32 -> bf16 (both steps RNE). Every
value is a pure function of (seed, tensor id, element index), so a row subset drawn on the
CPU equals the same rows drawn on the GPU (integer hashing is exact on both; the fp64
log/cos may differ in the last ulp between devices, which changes a bf16 value only when it
sits within 2^-44 relative of a rounding boundary).

Workload shapes follow the pages' `_o_proj` at DeepSeek-V4.1-Flash TP1 ("8 groups x 4096 ->
1024, wo_b 8192 -> 5120", page "[Perf][DSv4.1] MegaAttn: wo_a writes wo_b's MXFP8 input",
Validation) and the RMSNorm producer of page "[Perf][DSv4.1] Keep activations MXFP8 between
DeepGEMM kernels" (Purpose). "N(0, s)" is read as standard deviation s.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import torch

GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK64 = (1 << 64) - 1

# tensor ids (stream selectors)
TID_O = 1
TID_O_GROUP = 2
TID_WA = 3
TID_WB = 4
TID_QX = 10
TID_QX_GROUP = 11
TID_QX_ELEM = 12
TID_RMS_X = 20
TID_RMS_GAMMA = 21
TID_RMS_OUTLIER = 22
TID_WQKV = 30
TID_SQ_A, TID_SQ_B = 40, 41  # the square 8192^3 GEMM of the bench sweep

# DeepSeek-V4.1 _o_proj shapes at TP1
G, NA, KA, NB = 8, 1024, 4096, 5120
KB = G * NA
RMS_H = 5120
RMS_EPS = 1e-6


# ---- reference (pure Python int) SplitMix64 ------------------------------------------------
def mix64_int(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * _M1) & _MASK64
    z = ((z ^ (z >> 27)) * _M2) & _MASK64
    return z ^ (z >> 31)


def splitmix64_sequence(seed: int, n: int) -> list:
    """The first n outputs of a SplitMix64 generator seeded with ``seed`` (pure Python)."""
    out, s = [], seed & _MASK64
    for _ in range(n):
        s = (s + GOLDEN) & _MASK64
        out.append(mix64_int(s))
    return out


def stream_key(seed: int, tid: int) -> int:
    return mix64_int(((seed & 0xFFFFFFFF) << 32) ^ (tid & 0xFFFFFFFF) ^ GOLDEN)


# ---- torch (int64, wrapping) SplitMix64 ------------------------------------------------------
def _i64(c: int) -> int:
    c &= _MASK64
    return c - (1 << 64) if c >= (1 << 63) else c


def _srl(z: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def hash64(key: int, idx: torch.Tensor) -> torch.Tensor:
    """mix64(key + (idx + 1) * GOLDEN) on int64 tensors (two's-complement wraparound)."""
    z = (idx + 1) * _i64(GOLDEN) + _i64(key)
    z = (z ^ _srl(z, 30)) * _i64(_M1)
    z = (z ^ _srl(z, 27)) * _i64(_M2)
    return z ^ _srl(z, 31)


def uniform(key: int, idx: torch.Tensor) -> torch.Tensor:
    """fp64 uniforms in (0, 1): (top 53 bits + 0.5) * 2^-53."""
    h = _srl(hash64(key, idx), 11)
    return (h.to(torch.float64) + 0.5) * (2.0 ** -53)


def normal(key: int, idx: torch.Tensor) -> torch.Tensor:
    """fp64 standard normals, Box-Muller on the uniforms of counters 2i and 2i+1."""
    u1 = uniform(key, 2 * idx)
    u2 = uniform(key, 2 * idx + 1)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def _to_bf16(x64: torch.Tensor) -> torch.Tensor:
    return x64.to(torch.float32).to(torch.bfloat16)


def _bits_to_bf16(bits: torch.Tensor) -> torch.Tensor:
    """int32 tensor of 16-bit patterns in [0, 0xFFFF] -> bf16 tensor with those bits."""
    signed = bits - ((bits >= 0x8000).to(bits.dtype) << 16)
    return signed.to(torch.int16).view(torch.bfloat16)


def _row_index(rows: Optional[torch.Tensor], nrows: int, ncols: int, device) -> torch.Tensor:
    if rows is None:
        rows = torch.arange(nrows, dtype=torch.int64, device=device)
    rows = rows.to(device=device, dtype=torch.int64)
    cols = torch.arange(ncols, dtype=torch.int64, device=device)
    return rows[:, None] * ncols + cols[None, :]


def _chunked_rows(nrows: int, ncols: int, rows: Optional[torch.Tensor], device, fn, out_dtype):
    """Evaluate fn(idx[r0:r1]) over row chunks to bound temporary memory."""
    if rows is None:
        rows = torch.arange(nrows, dtype=torch.int64, device=device)
    rows = rows.to(device=device, dtype=torch.int64)
    out = torch.empty((rows.numel(), ncols), dtype=out_dtype, device=device)
    step = max(1, (1 << 25) // max(ncols, 1))
    for r0 in range(0, rows.numel(), step):
        r1 = min(rows.numel(), r0 + step)
        out[r0:r1] = fn(_row_index(rows[r0:r1], nrows, ncols, device), rows[r0:r1])
    return out


def normal_bf16(seed: int, tid: int, nrows: int, ncols: int, std: float, rows=None,
                device="cpu") -> torch.Tensor:
    key = stream_key(seed, tid)
    return _chunked_rows(nrows, ncols, rows, device,
                         lambda idx, _r: _to_bf16(normal(key, idx) * std), torch.bfloat16)


# ---- _o_proj inputs ------------------------------------------------------------------------
def _uniform_int(bits16: torch.Tensor, n: int) -> torch.Tensor:
    """Map 16 random bits to an integer in [0, n) by multiply-shift (no int64 modulo)."""
    return ((bits16 & 0xFFFF) * n) >> 16


def _group_index(r: torch.Tensor, ngroups: int) -> torch.Tensor:
    """[R, ngroups] global indices of the 32-element groups of rows r."""
    return r[:, None] * ngroups + torch.arange(ngroups, dtype=torch.int64, device=r.device)[None, :]


def o_proj_activation(seed: int, T: int, rows=None, device="cpu") -> torch.Tensor:
    """Attention output o, bf16 [T, G*KA] ~ N(0, 1); 1% of the 32-element groups (chosen by a
    hash) are multiplied by 2^k with k uniform in [-8, 8]."""
    key = stream_key(seed, TID_O)
    gkey = stream_key(seed, TID_O_GROUP)
    ncols = G * KA
    ng = ncols // 32

    def fn(idx, r):
        v = _to_bf16(normal(key, idx)).to(torch.float32).view(idx.shape[0], ng, 32)
        gidx = _group_index(r, ng)
        pick = uniform(gkey, 2 * gidx) < 0.01
        k = _uniform_int(_srl(hash64(gkey, 2 * gidx + 1), 40), 17) - 8
        scale = torch.where(pick, torch.exp2(k.to(torch.float32)), torch.ones_like(k, dtype=torch.float32))
        return (v * scale[:, :, None]).to(torch.bfloat16).view(idx.shape[0], ncols)

    return _chunked_rows(T, ncols, rows, device, fn, torch.bfloat16)


def wo_a_weight(seed: int, device="cpu") -> torch.Tensor:
    """wo_a, bf16 [G*NA, KA] = [8*1024, 4096] ~ N(0, 1/sqrt(4096))."""
    return normal_bf16(seed, TID_WA, G * NA, KA, 1.0 / math.sqrt(KA), device=device)


def wo_b_weight(seed: int, device="cpu") -> torch.Tensor:
    """wo_b, bf16 [NB, G*NA] = [5120, 8192] ~ N(0, 1/sqrt(8192))."""
    return normal_bf16(seed, TID_WB, NB, KB, 1.0 / math.sqrt(KB), device=device)


# The down-projection that consumes RMSNorm's MXFP8 y ("fused_wqa_wkv"). The pages do not give
# its width; 2048 output features (a multiple of the 128-row weight tile) stand in for it.
WQKV_N = 2048


def wqa_wkv_weight(seed: int, N: int = WQKV_N, H: int = RMS_H, device="cpu") -> torch.Tensor:
    """fused_wqa_wkv stand-in, bf16 [N, H] ~ N(0, 1/sqrt(H))."""
    return normal_bf16(seed, TID_WQKV, N, H, 1.0 / math.sqrt(H), device=device)


# ---- standalone quantizer input ----------------------------------------------------------
# Hand-listed edge groups (bf16 bit patterns) placed in row 0: zeros of both signs, the
# largest finite bf16, subnormals, the smallest normal, values straddling 448 and the
# scale-rule boundary (mantissa 96 vs 97), and E4M3 rounding ties.
def _edge_groups() -> list:
    g = []
    def bits(v: float) -> int:
        return int(torch.tensor([v], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item()) & 0xFFFF
    g.append([0x0000] * 16 + [0x8000] * 16)                       # +0 / -0
    g.append([0x7F7F, 0xFF7F] + [0x3F80] * 30)                    # +-max finite bf16
    g.append([0x0001, 0x8001, 0x007F, 0x807F] * 8)                # subnormals only
    g.append([0x0080, 0x8080] + [0x0001] * 30)                    # min normal + subnormals
    g.append([bits(448.0), bits(-448.0)] + [bits(1.0)] * 30)      # amax exactly 448
    g.append([bits(450.0)] + [bits(-1.0)] * 31)                   # first bf16 above 448
    g.append([bits(1.75)] + [bits(1.0 + (2 * j + 1) / 16) for j in range(8)] * 3 + [bits(0.5)] * 7)
    g.append([bits(1.7578125)] + [bits((1.0 + (2 * j + 1) / 16) * 2.0) for j in range(8)] * 3 + [bits(-0.25)] * 7)
    g.append([bits(2.0 ** -6 * (7.5 / 8))] * 8 + [bits(2.0 ** -10)] * 8 + [bits(1.75)] + [bits(-2.0 ** -9 * 1.5)] * 15)
    g.append([bits(2.0 ** -127)] * 31 + [bits(2.0 ** -133)])      # subnormal amax
    g.append([bits(3.0 * 2.0 ** 120)] + [bits(1.0)] * 31)          # huge amax, ones underflow
    g.append([bits(-(2.0 ** 100))] + [bits(2.0 ** -30)] * 31)
    return g


EDGE_GROUPS = _edge_groups()


def quantizer_input(seed: int, T: int, K: int = KB, rows=None, device="cpu") -> torch.Tensor:
    """bf16 [T, K]: N(0,1) with every 32-element group scaled by 2^k (k uniform in [-20, 20]),
    plus hash-selected special groups -- 1% all-zero (mixed signs of zero), 1% all-subnormal,
    1% mixed subnormal/normal, 1% holding one +-large finite value, 0.5% on the scale-rule and
    rounding boundaries (amax mantissa 96 or 97, other elements on E4M3 midpoints) -- and the
    hand-listed edge groups in row 0."""
    key = stream_key(seed, TID_QX)
    gkey = stream_key(seed, TID_QX_GROUP)
    ekey = stream_key(seed, TID_QX_ELEM)
    assert K % 32 == 0
    ng = K // 32
    edge_list = [b_ for grp in EDGE_GROUPS for b_ in grp][: K]

    def fn(idx, r):
        R = idx.shape[0]
        n = normal(key, idx).to(torch.float32).view(R, ng, 32)
        gidx = _group_index(r, ng)                                   # [R, ng]
        cls = uniform(gkey, 4 * gidx)[:, :, None]
        gh = _srl(hash64(gkey, 4 * gidx + 2), 8)                     # 56 per-group bits
        k = (_uniform_int(gh >> 24, 41) - 20).to(torch.float32)[:, :, None]
        big_pos = (gh & 31)[:, :, None]
        p = (_uniform_int(gh >> 5, 161) - 80).to(torch.int32)[:, :, None]
        mant = torch.where(((gh >> 21) & 1) == 1, 97, 96).to(torch.int32)[:, :, None]
        eh = _srl(hash64(ekey, idx), 8).view(R, ng, 32)               # 56 per-element bits
        pos = torch.arange(32, dtype=torch.int64, device=idx.device)[None, None, :]
        sign = ((eh & 1) << 15).to(torch.int32)
        base = (n * torch.exp2(k)).to(torch.bfloat16).view(torch.int16).to(torch.int32) & 0xFFFF
        zero = sign                                                   # +0 or -0
        sub = sign | torch.clamp((eh >> 1) & 127, min=1).to(torch.int32)  # exponent field 0
        mixed = torch.where(((eh >> 9) & 1) == 1, sub, base)
        big = sign | (0x7F00 + ((eh >> 1) & 127)).to(torch.int32)
        withbig = torch.where(pos == big_pos, big, base)
        # boundary groups: amax = (1 + m/128) * 2^p with m in {96, 97}; the other elements are
        # E4M3 midpoints (1 + (2j+1)/16) * 2^(b + p - 8), b in [-6, 7]
        amax_bits = ((p + 127) << 7) | mant
        jj = ((eh >> 1) & 7).to(torch.int32)
        b = (_uniform_int(eh >> 4, 14) - 6).to(torch.int32)
        tie_bits = ((b + p - 8 + 127) << 7) | ((2 * jj + 1) << 3)
        bnd = torch.where(pos == big_pos, amax_bits, tie_bits) | sign
        out = base
        out = torch.where(cls < 0.045, bnd, out)
        out = torch.where(cls < 0.04, withbig, out)
        out = torch.where(cls < 0.03, mixed, out)
        out = torch.where(cls < 0.02, sub, out)
        out = torch.where(cls < 0.01, zero, out)
        out = out.view(R, K)
        first = torch.nonzero(r == 0).flatten()
        if first.numel():
            edge = torch.tensor(edge_list, dtype=torch.int32, device=idx.device)
            out[first, : edge.numel()] = edge
        return _bits_to_bf16(out)

    return _chunked_rows(T, K, rows, device, fn, torch.bfloat16)


# ---- RMSNorm producer input ----------------------------------------------------------------
def rmsnorm_outlier_channels(seed: int, H: int = RMS_H, count: int = 5) -> list:
    """`count` distinct channels of H (0.1% of 5120 = 5), chosen by hash order."""
    key = stream_key(seed, TID_RMS_OUTLIER)
    h = hash64(key, torch.arange(H, dtype=torch.int64))
    order = torch.argsort(_srl(h, 1))
    return sorted(int(c) for c in order[:count])


def rmsnorm_input(seed: int, T: int, H: int = RMS_H, rows=None, device="cpu") -> torch.Tensor:
    """x bf16 [T, H] ~ N(0, 3) with 0.1% of the channels multiplied by 50 in every row."""
    key = stream_key(seed, TID_RMS_X)
    ch = torch.zeros(H, dtype=torch.bool)
    ch[rmsnorm_outlier_channels(seed, H, max(1, H // 1000))] = True
    ch = ch.to(device)

    def fn(idx, _r):
        v = normal(key, idx) * 3.0
        col = idx % H
        v = torch.where(ch[col], v * 50.0, v)
        return _to_bf16(v)

    return _chunked_rows(T, H, rows, device, fn, torch.bfloat16)


def rmsnorm_gamma(seed: int, H: int = RMS_H, device="cpu") -> torch.Tensor:
    """gamma bf16 [H] ~ N(1, 0.1)."""
    key = stream_key(seed, TID_RMS_GAMMA)
    idx = torch.arange(H, dtype=torch.int64, device=device)
    return _to_bf16(1.0 + 0.1 * normal(key, idx))


def sample_rows(seed: int, T: int, n_random: int = 256, tile: int = 128) -> torch.Tensor:
    """Row subset for full-size checks: the first and last 128-row tiles plus n_random seeded
    rows in between (sorted, unique)."""
    first = list(range(min(tile, T)))
    last_start = ((T - 1) // tile) * tile
    last = list(range(last_start, T))
    key = stream_key(seed, 99)
    h = _srl(hash64(key, torch.arange(n_random, dtype=torch.int64)), 8) % max(T, 1)
    rows = sorted(set(first) | set(last) | set(int(v) for v in h))
    return torch.tensor(rows, dtype=torch.int64)


def bf16_bits(x: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    return x.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
