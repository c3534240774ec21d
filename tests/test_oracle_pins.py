"""Pins for the CPU oracle, against what the format definitions and mathematics fix.

None of these tests re-derives the oracle's own formulas: each compares the oracle with an
independent statement of the same fact -- torch's float8_e4m3fn codec (a library), brute-force
nearest-grid and minimal-exponent searches, exact rational arithmetic, numpy's einsum and
torch's rms_norm, closed forms and invariants.

Format facts pinned here come from the OCP FP8 E4M3 definition that the pages name as
"MXFP8 / OCP FP8" (page "[Perf][DSv4.1] Keep activations MXFP8 between DeepGEMM kernels",
review) and from the scale rule: the smallest power of two 2^e with amax / 2^e <= 448.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN_DIR = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------------------------
# independent helpers
# ---------------------------------------------------------------------------------------------
def torch_e4m3_table() -> np.ndarray:
    """Decode of all 256 codes by torch's float8_e4m3fn (library codec)."""
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def all_finite_bf16_bits() -> np.ndarray:
    b = np.arange(65536, dtype=np.uint32)
    exp = (b >> 7) & 0xFF
    return b[exp != 0xFF].astype(np.uint16)  # 65280 patterns (both zeros included)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def brute_force_e4m3(q: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 value by search over torch's decode table; equidistant -> even
    code; |q| >= 448 -> +-448; the sign of a zero result follows q."""
    table = torch_e4m3_table()
    grid = table[:0x7F]                       # codes 0x00..0x7E, ascending, all finite
    assert np.all(np.diff(grid) > 0)
    a = np.abs(q)
    hi = np.clip(np.searchsorted(grid, a), 0, 0x7E)
    lo = np.clip(hi - 1, 0, 0x7E)
    d_lo = a - grid[lo]
    d_hi = grid[hi] - a
    pick = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    pick = np.where(a >= 448.0, 0x7E, pick)
    sign = np.signbit(q).astype(np.uint8) << 7
    return (pick.astype(np.uint8) | sign).astype(np.uint8)


def brute_force_min_exponent(amax: np.ndarray) -> np.ndarray:
    """Smallest integer e in [-127, 127] with amax <= 448 * 2^e (exact fp64 comparisons)."""
    e_best = np.full(amax.shape, 999, np.int64)
    for e in range(-127, 128):
        ok = (amax <= np.ldexp(448.0, e)) & (e_best == 999)
        e_best[ok] = e
    return e_best


# ---------------------------------------------------------------------------------------------
# E4M3 decode (C1)
# ---------------------------------------------------------------------------------------------
def test_e4m3_decode_all_codes_match_library(oracle):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch_e4m3_table()
    nan_o, nan_r = np.isnan(ours), np.isnan(ref)
    assert np.array_equal(nan_o, nan_r)
    assert set(np.nonzero(nan_o)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan_o], ref[~nan_r])
    assert np.array_equal(np.signbit(ours[~nan_o]), np.signbit(ref[~nan_r]))


def test_e4m3_special_values(oracle):
    d = oracle.e4m3_decode(np.array([0x7E, 0x08, 0x01, 0x00, 0x80, 0xFE, 0x38], np.uint8))
    assert d[0] == 448.0
    assert d[1] == 2.0 ** -6
    assert d[2] == 2.0 ** -9
    assert d[3] == 0.0 and not np.signbit(d[3])
    assert d[4] == 0.0 and np.signbit(d[4])
    assert d[5] == -448.0
    assert d[6] == 1.0


def test_e4m3_roundtrip_and_monotone(oracle):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    assert codes.size == 254
    vals = oracle.e4m3_decode(codes)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)


# ---------------------------------------------------------------------------------------------
# E4M3 encode (C2)
# ---------------------------------------------------------------------------------------------
def test_e4m3_encode_every_bf16_direct(oracle):
    x = bf16_bits_to_f64(all_finite_bf16_bits())
    assert np.array_equal(oracle.e4m3_encode(x), brute_force_e4m3(x))


def test_e4m3_encode_every_bf16_at_every_scale(oracle):
    """Every finite bf16 value x times every scale 2^-e, e in [-127, 120] (16.2 M cases)."""
    x = bf16_bits_to_f64(all_finite_bf16_bits())
    for e0 in range(-127, 121, 31):
        es = np.arange(e0, min(e0 + 31, 121))
        q = np.ldexp(x[None, :], -es[:, None]).reshape(-1)
        assert np.array_equal(oracle.e4m3_encode(q), brute_force_e4m3(q)), f"e in {es[0]}..{es[-1]}"


def test_e4m3_encode_hand_listed_ties(oracle):
    cases = [
        (1.0625, 0x38),              # tie between 1.0 (m=0) and 1.125 (m=1) -> even 1.0
        (1.1875, 0x3A),              # tie between 1.125 (m=1) and 1.25 (m=2) -> 1.25
        (0.9375 * 2.0 ** -6, 0x08),  # subnormal/normal midpoint -> 2^-6 (even code 0x08)
        (2.0 ** -10, 0x00),          # half of the smallest subnormal -> 0
        (-(2.0 ** -10), 0x80),       # sign of a zero result follows q
        (3 * 2.0 ** -10, 0x02),      # 1.5 * 2^-9 -> 2 * 2^-9 (even)
        (464.0, 0x7E),               # saturates
        (1e30, 0x7E),
        (-1e30, 0xFE),
        (0.0, 0x00),
        (-0.0, 0x80),
    ]
    q = np.array([c[0] for c in cases])
    want = np.array([c[1] for c in cases], np.uint8)
    assert np.array_equal(oracle.e4m3_encode(q), want)
    assert np.array_equal(brute_force_e4m3(q), want)


def test_e4m3_encode_matches_library_cast_in_range(oracle):
    rng = np.random.default_rng(0)
    q = np.concatenate([rng.uniform(-448, 448, 200000),
                        rng.standard_normal(200000) * 2.0 ** rng.integers(-12, 8, 200000)])
    q = q.astype(np.float32).astype(np.float64)  # torch casts from fp32
    q = q[np.abs(q) <= 448.0]                    # torch's cast does not saturate above 464
    lib = torch.from_numpy(q.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(q), lib)


# ---------------------------------------------------------------------------------------------
# UE8M0 scale rule (C3)
# ---------------------------------------------------------------------------------------------
def test_ue8m0_every_bf16_amax(oracle):
    bits = all_finite_bf16_bits()
    bits = bits[bits < 0x8000]                      # non-negative amax values
    amax = bf16_bits_to_f64(bits)
    code = oracle.ue8m0_from_amax(amax).astype(np.int64)
    pos = amax > 0
    e_bf = brute_force_min_exponent(amax[pos])
    assert np.array_equal(code[pos] - 127, np.maximum(e_bf, -127))
    assert code[~pos].tolist() == [0]                # all-zero group -> smallest scale
    # invariants: amax / 2^e <= 448, and e minimal unless clamped at -127
    e = code[pos] - 127
    assert np.all(amax[pos] / np.ldexp(1.0, e) <= 448.0)
    unclamped = e > -127
    assert np.all(amax[pos][unclamped] / np.ldexp(1.0, e[unclamped] - 1) > 448.0)
    # closed form in the bf16 fields (E biased exponent, m 7-bit mantissa), derived by hand:
    # 448 = 1.75 * 2^8 and 1.75 is mantissa 96, so code = max(0, E - 8 + [m > 96]).
    E = (bits.astype(np.int64) >> 7) & 0xFF
    m = bits.astype(np.int64) & 0x7F
    assert np.array_equal(code, np.maximum(0, E - 8 + (m > 96)))
    assert code.max() == 247                         # never needs the upper clamp


# ---------------------------------------------------------------------------------------------
# group quantizer (C4)
# ---------------------------------------------------------------------------------------------
def _quantize_reference_python(xbits_row: np.ndarray):
    """Group quantize by brute force: minimal exponent by search, nearest code by search."""
    x = bf16_bits_to_f64(xbits_row)
    q = np.empty(x.size, np.uint8)
    sf = np.empty(x.size // 32, np.uint8)
    for g in range(x.size // 32):
        v = x[32 * g: 32 * g + 32]
        amax = np.max(np.abs(v))
        e = -127 if amax == 0 else max(int(brute_force_min_exponent(np.array([amax]))[0]), -127)
        sf[g] = e + 127
        q[32 * g: 32 * g + 32] = brute_force_e4m3(np.ldexp(v, -e))
    return q, sf


def test_quantize_matches_brute_force_on_edges(oracle):
    from mxfp8_activation_quant_gb300 import synth

    x = synth.bf16_bits(synth.quantizer_input(0, 4, K=1024))
    q, sf = oracle.quantize_bf16(x)
    for r in range(4):
        qr, sfr = _quantize_reference_python(x[r])
        assert np.array_equal(q[r], qr)
        assert np.array_equal(sf[r], sfr)


def test_quantize_edge_groups_by_hand(oracle):
    from mxfp8_activation_quant_gb300 import synth

    x = np.array(synth.EDGE_GROUPS, np.uint16).reshape(1, -1)
    q, sf = oracle.quantize_bf16(x)
    sf = sf[0]
    # group 0: zeros of both signs -> scale byte 0, codes 0x00 / 0x80
    assert sf[0] == 0 and set(q[0, :16]) == {0x00} and set(q[0, 16:32]) == {0x80}
    # group 1: amax = max bf16 = 1.9921875 * 2^127 -> mantissa 127 > 96 -> byte 254 - 8 + 1;
    # amax / 2^120 = 255 -> nearest E4M3 is 256 (exponent field 15, mantissa 0 = 0x78)
    assert sf[1] == 247 and q[0, 32] == 0x78 and q[0, 33] == 0xF8
    # group 4: amax exactly 448 -> 2^0, codes 448 -> 0x7E, 1.0 -> 0x38
    assert sf[4] == 127 and q[0, 128] == 0x7E and q[0, 129] == 0xFE and q[0, 130] == 0x38
    # group 5: amax 450 (> 448) -> 2^1: 450/2 = 225 -> nearest E4M3 224 (0x76)
    assert sf[5] == 128 and q[0, 160] == 0x76
    # group 9: subnormal amax -> byte 0, values * 2^127 land on E4M3 subnormals exactly
    assert sf[9] == 0


def test_quantize_dequant_error_bound(oracle):
    from mxfp8_activation_quant_gb300 import synth

    xb = synth.bf16_bits(synth.quantizer_input(1, 64, K=2048))
    q, sf = oracle.quantize_bf16(xb)
    x = bf16_bits_to_f64(xb)
    scale = np.ldexp(1.0, sf.astype(np.int64) - 127)
    deq = torch_e4m3_table()[q] * np.repeat(scale, 32, axis=1)
    # half an E4M3 ulp at the value's binade, in scaled units: ulp = 2^(max(E,-6) - 3)
    qv = np.abs(x) / np.repeat(scale, 32, axis=1)
    with np.errstate(divide="ignore"):
        binade = np.floor(np.log2(np.where(qv > 0, qv, 1.0)))
    ulp = np.ldexp(1.0, (np.maximum(binade, -6) - 3).astype(np.int64))
    err = np.abs(x - deq) / np.repeat(scale, 32, axis=1)
    assert np.all(err <= 0.5 * ulp + 0.0)
    assert np.all(qv <= 448.0)


# ---------------------------------------------------------------------------------------------
# scale layouts (C5)
# ---------------------------------------------------------------------------------------------
def test_128x4_layout_is_the_32x16B_warp_view(oracle):
    """A 128-row x 4-group tile viewed as 32 lines of 16 bytes: line i holds rows i, i+32,
    i+64, i+96, each as 4 consecutive group bytes (written here with numpy reshapes)."""
    rng = np.random.default_rng(3)
    M, Kg = 300, 12
    sf = rng.integers(0, 255, (M, Kg), dtype=np.uint8)
    buf = oracle.sf_to_128x4(sf)
    Mp, Gp = 384, 12
    pad = np.zeros((Mp, Gp), np.uint8)
    pad[:M, :Kg] = sf
    tiles = pad.reshape(Mp // 128, 128, Gp // 4, 4).transpose(0, 2, 1, 3)     # [rt, ct, 128, 4]
    view = tiles.reshape(Mp // 128, Gp // 4, 4, 32, 4).transpose(0, 1, 3, 2, 4)  # [rt, ct, i, q, c]
    assert np.array_equal(buf, view.reshape(-1))
    assert np.array_equal(oracle.sf_from_128x4(buf, M, Kg), sf)
    # one hand-computed position: row 33, group 5 of a 200 x 8 scale matrix
    s = np.zeros((200, 8), np.uint8)
    s[33, 5] = 7
    b = oracle.sf_to_128x4(s)
    assert b.size == 256 * 8 and np.nonzero(b)[0].tolist() == [512 + 16 + 4 + 1]


def test_128x4_padding_is_zero(oracle):
    sf = np.full((5, 3), 0xAB, np.uint8)
    buf = oracle.sf_to_128x4(sf)
    assert buf.size == 128 * 4
    assert int((buf == 0xAB).sum()) == 15 and int((buf == 0).sum()) == 512 - 15


def test_packed_i32_roundtrip_and_byte_order(oracle):
    rng = np.random.default_rng(4)
    M, Kg = 7, 8
    sf = rng.integers(0, 255, (M, Kg), dtype=np.uint8)
    p = oracle.sf_pack_i32(sf)
    assert p.shape == (2, 8)                       # Kg/4 words x ceil(M/4)*4 rows
    assert np.all(p[:, 7] == 0)                    # padding row
    assert p[1, 3] == int.from_bytes(bytes(sf[3, 4:8].tolist()), "little")
    assert np.array_equal(oracle.sf_unpack_i32(p, M, Kg), sf)


# ---------------------------------------------------------------------------------------------
# GEMMs (C6)
# ---------------------------------------------------------------------------------------------
def _frac_e4m3(code: int) -> Fraction:
    v = torch_e4m3_table()[code]
    return Fraction(float(v))


def test_gemm_bruteforce_exact_rationals(oracle):
    rng = np.random.default_rng(5)
    T, K, N = 3, 64, 5
    aq = rng.integers(0, 256, (T, K), dtype=np.uint8)
    bq = rng.integers(0, 256, (N, K), dtype=np.uint8)
    aq[(aq & 0x7F) == 0x7F] = 0x11
    bq[(bq & 0x7F) == 0x7F] = 0x22
    asf = rng.integers(120, 134, (T, K // 32), dtype=np.uint8)
    bsf = rng.integers(120, 134, (N, K // 32), dtype=np.uint8)
    C = oracle.gemm_nt(oracle.dequant(aq, asf), oracle.dequant(bq, bsf))
    for t in range(T):
        for n in range(N):
            s = Fraction(0)
            for k in range(K):
                s += (_frac_e4m3(aq[t, k]) * Fraction(2) ** (int(asf[t, k // 32]) - 127)
                      * _frac_e4m3(bq[n, k]) * Fraction(2) ** (int(bsf[n, k // 32]) - 127))
            assert C[t, n] == float(s), (t, n)     # exact: the terms span < 53 bits


def test_gemm_identity_weights_reduce_to_copy(oracle):
    """Unit scales and an identity wa make the einsum a copy of o's group slice."""
    rng = np.random.default_rng(6)
    G_, Na, Ka, T = 2, 32, 32, 4
    oq = rng.integers(0, 0x7E, (T, G_ * Ka), dtype=np.uint8)
    osf = np.full((T, G_ * Ka // 32), 127, np.uint8)
    one = oracle.e4m3_encode(np.array([1.0]))[0]
    waq = np.zeros((G_ * Na, Ka), np.uint8)
    for g in range(G_):
        waq[g * Na + np.arange(Na), np.arange(Ka)] = one
    wasf = np.full((G_ * Na, Ka // 32), 127, np.uint8)
    z = oracle.einsum_wo_a(oracle.dequant(oq, osf), oracle.dequant(waq, wasf), G_)
    assert np.array_equal(z, torch_e4m3_table()[oq])


def test_einsum_matches_numpy(oracle):
    rng = np.random.default_rng(7)
    T, G_, Na, Ka = 3, 4, 16, 64
    o = rng.standard_normal((T, G_ * Ka))
    wa = rng.standard_normal((G_ * Na, Ka))
    z = oracle.einsum_wo_a(o, wa, G_)
    ref = np.einsum("tgk,gnk->tgn", o.reshape(T, G_, Ka), wa.reshape(G_, Na, Ka)).reshape(T, G_ * Na)
    np.testing.assert_allclose(z, ref, rtol=1e-12, atol=1e-12)
    C = oracle.gemm_nt(o, rng.standard_normal((5, G_ * Ka)))
    assert C.shape == (T, 5)


def test_gemm_matches_numpy_matmul(oracle):
    rng = np.random.default_rng(8)
    A = rng.standard_normal((9, 96))
    B = rng.standard_normal((13, 96))
    np.testing.assert_allclose(oracle.gemm_nt(A, B), A @ B.T, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------------------------
# bf16 rounding and RMSNorm (C7)
# ---------------------------------------------------------------------------------------------
def test_bf16_round_nearest_even_bruteforce(oracle):
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.standard_normal(20000) * 2.0 ** rng.integers(-140, 120, 20000),
                        [0.0, -0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 2.0 ** -134, 3 * 2.0 ** -134]])
    got = oracle.bf16_round(x)
    vals = bf16_bits_to_f64(all_finite_bf16_bits())
    vals = np.unique(vals)                       # ascending, -0 and +0 merged
    bits_of = {}
    for b in all_finite_bf16_bits():
        bits_of.setdefault(float(bf16_bits_to_f64(np.array([b]))[0]), []).append(int(b))
    hi = np.clip(np.searchsorted(vals, x), 0, vals.size - 1)
    lo = np.clip(hi - 1, 0, vals.size - 1)
    for i in range(x.size):
        a, b_ = vals[lo[i]], vals[hi[i]]
        da, db = abs(x[i] - a), abs(b_ - x[i])
        if da < db:
            v = a
        elif db < da:
            v = b_
        else:  # tie: the candidate with an even last significand bit
            ca = min(bits_of[float(a)])
            v = a if (ca & 1) == 0 else b_
        bits = [bb for bb in bits_of[float(v)] if (v != 0.0) or ((bb >> 15) == int(np.signbit(x[i])))]
        assert got[i] == bits[0], (x[i], got[i], bits)
    # fp32-representable values: torch's fp32 -> bf16 cast is a single RNE rounding
    f = (rng.standard_normal(50000) * 10).astype(np.float32)
    lib = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_round(f.astype(np.float64)), lib)


def test_rmsnorm_closed_forms(oracle):
    H = 256
    one = np.full(H, 0x3F80, np.uint16)  # gamma = 1
    c = 3.0
    x = np.full((1, H), 0x4040, np.uint16)  # 3.0
    y = oracle.rmsnorm(x, one, 1e-6)
    np.testing.assert_allclose(y, c / np.sqrt(c * c + 1e-6), rtol=1e-15)
    x1 = np.zeros((1, H), np.uint16)
    x1[0, 17] = 0x4000  # 2.0: mean of squares 4/H
    y1 = oracle.rmsnorm(x1, one, 0.0)
    assert y1[0, 17] == pytest.approx(np.sqrt(H), rel=1e-15) and np.count_nonzero(y1) == 1


def test_rmsnorm_matches_library(oracle):
    from mxfp8_activation_quant_gb300 import synth

    x = synth.rmsnorm_input(0, 8, H=512)
    g = synth.rmsnorm_gamma(0, H=512)
    y = oracle.rmsnorm(synth.bf16_bits(x), synth.bf16_bits(g), 1e-6)
    ref = torch.nn.functional.rms_norm(x.double(), (512,), weight=g.double(), eps=1e-6).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=0)


# ---------------------------------------------------------------------------------------------
# the chain composes the pinned steps
# ---------------------------------------------------------------------------------------------
def test_o_proj_chain_small(oracle):
    rng = np.random.default_rng(10)
    T, G_, Na, Ka, Nb = 5, 2, 128, 64, 96
    def mx(rows, cols, std):
        x = torch.from_numpy(rng.standard_normal((rows, cols)) * std).float().to(torch.bfloat16)
        return oracle.quantize_bf16(x.view(torch.int16).numpy().view(np.uint16))
    oq, osf = mx(T, G_ * Ka, 1.0)
    waq, wasf = mx(G_ * Na, Ka, 0.1)
    wbq, wbsf = mx(Nb, G_ * Na, 0.1)
    r = oracle.o_proj_chain(oq, osf, waq, wasf, wbq, wbsf, G_)
    o = oracle.dequant(oq, osf).reshape(T, G_, Ka)
    wa = oracle.dequant(waq, wasf).reshape(G_, Na, Ka)
    z = np.einsum("tgk,gnk->tgn", o, wa).reshape(T, G_ * Na)
    np.testing.assert_allclose(r["z_ref"], z, rtol=1e-12, atol=1e-12)
    zq, zsf = oracle.quantize_bf16(r["z_bf16"])
    assert np.array_equal(zq, r["zq"]) and np.array_equal(zsf, r["zsf"])
    out = oracle.dequant(zq, zsf) @ oracle.dequant(wbq, wbsf).T
    np.testing.assert_allclose(r["out_ref"], out, rtol=1e-12, atol=1e-12)
    # bf16 rounding of z alone stays within half an ulp: 2^-8 relative (7 stored mantissa bits)
    zb = bf16_bits_to_f64(r["z_bf16"])
    assert np.all(np.abs(zb - z) <= np.abs(z) * 2.0 ** -8)


def test_golden_fixtures(oracle):
    """Values fixed by the format definitions, stored under tests/golden with citations."""
    with open(os.path.join(GOLDEN_DIR, "e4m3_ue8m0_points.json")) as f:
        g = json.load(f)
    for row in g["e4m3_encode"]:
        assert int(oracle.e4m3_encode(np.array([row["q"]]))[0]) == row["code"], row
    for row in g["ue8m0"]:
        assert int(oracle.ue8m0_from_amax(np.array([row["amax"]]))[0]) == row["byte"], row
