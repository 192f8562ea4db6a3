"""Pins for the oracle's number formats (CPU only).

Each check compares the oracle with something other than itself: the
formats' closed forms written out as literal values, brute force over every
code and every midpoint, the UE8M0 identity printed on the vllm.models.
qwen4_exp.nvidia.mega_moe page (``_requantize``: a power-of-two fp32 scale's
exponent bits are the UE8M0 byte), and hand-worked blocks in tests/golden/.
"""
import json
import math
import os
import struct

import numpy as np
import pytest

from oracle import formats as F


# ----------------------------------------------------------------------------- decode tables

def test_e2m1_table_literal():
    # OCP MX E2M1: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; bit 3 is the sign
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert F.E2M1_TABLE[:8].tolist() == mags
    assert F.E2M1_TABLE[8:].tolist() == [-m for m in mags]
    assert math.copysign(1.0, F.E2M1_TABLE[8]) == -1.0


def test_e4m3_table_landmarks():
    # landmark codes of E4M3 (fn), values written out by hand
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
             0x38: 1.0, 0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x70: 128.0, 0x78: 256.0,
             0x7E: 448.0, 0x80: -0.0, 0xB8: -1.0, 0xFE: -448.0}
    for c, v in cases.items():
        assert F.E4M3_TABLE[c] == v, hex(c)
    assert np.isnan(F.E4M3_TABLE[0x7F]) and np.isnan(F.E4M3_TABLE[0xFF])
    assert np.isnan(F.E4M3_TABLE).sum() == 2


def test_e4m3_table_brute_force_against_fp16():
    # every finite E4M3 value is an fp16 value: rebuild it from fp16 bits
    # (fp16 exponent bias 15 vs 7: shift mantissa by 7, add 8 to the exponent)
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        s, e, m = c >> 7, (c >> 3) & 0xF, c & 7
        if e == 0:
            ref = m * 2.0 ** -9
        else:
            bits = ((e + 8) << 10) | (m << 7)
            ref = float(np.frombuffer(struct.pack("<H", bits), dtype=np.float16)[0])
        assert abs(F.E4M3_TABLE[c]) == ref
        assert bool(np.signbit(F.E4M3_TABLE[c])) == bool(s)


def test_ue8m0_matches_page_identity():
    # vllm.models.qwen4_exp.nvidia.mega_moe, _requantize: UE8M0 byte b is the fp32 bit
    # pattern b << 23 (for b >= 1; b == 0 would be fp32 zero, not 2^-127)
    for b in range(1, 255):
        as_f32 = struct.unpack("<f", struct.pack("<I", b << 23))[0]
        assert F.UE8M0_TABLE[b] == as_f32
    assert F.UE8M0_TABLE[0] == 2.0 ** -127
    assert np.isnan(F.UE8M0_TABLE[255])


# ----------------------------------------------------------------------------- encoders

def test_e4m3_round_trip_every_code():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    assert np.array_equal(F.e4m3_encode(F.E4M3_TABLE[codes]), codes)


def test_e2m1_round_trip_every_code():
    codes = np.arange(16, dtype=np.uint8)
    assert np.array_equal(F.e2m1_encode(F.E2M1_TABLE[codes]), codes)


@pytest.mark.parametrize("table,enc,top,sign", [
    (F.E4M3_TABLE, F.e4m3_encode, 0x7E, 0x80),
    (F.E2M1_TABLE, F.e2m1_encode, 0x7, 0x8),
])
def test_midpoints_tie_to_even_and_neighbours(table, enc, top, sign):
    for c in range(top):
        a, b = table[c], table[c + 1]
        mid = (a + b) / 2
        even = c if c % 2 == 0 else c + 1
        assert enc(mid) == even
        assert enc(-mid) == even | sign
        assert enc(np.nextafter(mid, -np.inf)) == c
        assert enc(np.nextafter(mid, np.inf)) == c + 1


def test_e2m1_tie_table():
    # ties: 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4
    vals = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    want = [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]
    assert F.E2M1_TABLE[F.e2m1_encode(vals)].tolist() == want


def test_saturation():
    assert F.e4m3_encode([448.0, 449.0, 464.0, 1e30, -1e30]).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE]
    assert F.e2m1_encode([6.0, 6.5, 1e9, -7.0]).tolist() == [7, 7, 7, 15]
    with pytest.raises(ValueError):
        F.e4m3_encode([np.nan])


def test_signed_zero():
    assert F.e4m3_encode([0.0, -0.0, -1e-9]).tolist() == [0x00, 0x80, 0x80]
    assert F.e2m1_encode([0.0, -0.0, -0.1]).tolist() == [0x0, 0x8, 0x8]


def test_e2m1_pack_order():
    packed = F.pack_e2m1(np.array([[1, 2, 3, 4]], dtype=np.uint8))
    assert packed.tolist() == [[0x21, 0x43]]
    assert F.unpack_e2m1(packed).tolist() == [[1, 2, 3, 4]]


def test_bf16_round_brute_force():
    rng = np.random.default_rng(1)
    v = rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))
    r = F.bf16_round(v)
    # r is a bf16 value (low 16 fp32 bits zero) and no bf16 value is nearer
    bits = r.astype(np.float32).view(np.uint32)
    assert np.all(bits & 0xFFFF == 0)
    up = (bits + (1 << 16)).view(np.float32).astype(np.float64)
    dn = (bits - (1 << 16)).view(np.float32).astype(np.float64)
    assert np.all(np.abs(v - r) <= np.abs(v - up))
    assert np.all(np.abs(v - r) <= np.abs(v - dn))
    # exact midpoint ties to an even mantissa
    one = 1.0 + 2.0 ** -8
    assert F.bf16_round(one) == 1.0 and F.bf16_round(1.0 + 3 * 2.0 ** -8) == 1.0 + 2 * 2.0 ** -7


# ----------------------------------------------------------------------------- MXFP8

def test_ue8m0_exponent_exact_powers():
    n = np.arange(-40, 41)
    amax = np.ldexp(448.0, n)
    assert np.array_equal(F.ue8m0_exponent(amax), n)
    assert np.array_equal(F.ue8m0_exponent(np.nextafter(amax, np.inf)), n + 1)
    assert np.array_equal(F.ue8m0_exponent(np.nextafter(amax, -np.inf)), n)
    assert F.ue8m0_exponent(0.0) == 0


def test_ue8m0_exponent_matches_frexp_route():
    # independent route: amax = f * 2^p with f in [0.5, 1); 448 = 0.875 * 2^9
    rng = np.random.default_rng(2)
    amax = np.exp(rng.uniform(-30, 30, 5000))
    for a, e in zip(amax, F.ue8m0_exponent(amax)):
        f, p = math.frexp(a)
        want = p - 9 if f <= 0.875 else p - 8
        assert e == want


def test_mxfp8_scale_is_page_exponent_bits():
    # the power-of-two fp32 scale's exponent field is the UE8M0 byte
    rng = np.random.default_rng(3)
    x = rng.standard_normal((8, 64)) * np.exp(rng.uniform(-10, 10, (8, 1)))
    _, sf = F.mxfp8_quantize(x)
    e = F.ue8m0_exponent(np.abs(x.reshape(8, 2, 32)).max(-1))
    scale = np.ldexp(1.0, e).astype(np.float32)
    assert np.array_equal((scale.view(np.uint32) >> 23).astype(np.uint8), sf)


def test_mxfp8_error_bound_and_range():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((16, 256))
    codes, sf = F.mxfp8_quantize(x)
    deq = F.mxfp8_dequantize(codes, sf)
    scale = F.UE8M0_TABLE[sf].repeat(32, axis=1)
    y = x / scale                                     # exact; |y| <= 448
    assert np.abs(y).max() <= 448
    # E4M3 spacing around |y|: 2^(floor(log2|y|)-3) for normals, 2^-9 below 2^-6
    ulp = np.where(np.abs(y) >= 2 ** -6, np.ldexp(1.0, np.floor(np.log2(np.abs(y) + 1e-300)).astype(int) - 3), 2.0 ** -9)
    assert np.all(np.abs(deq - x) <= 0.5 * ulp * scale + 1e-300)
    # each block's amax lands in (224, 448] after scaling (for nonzero blocks)
    amax_scaled = np.abs(y.reshape(16, 8, 32)).max(-1)
    assert np.all((amax_scaled > 224) & (amax_scaled <= 448))


def test_mxfp8_zero_block():
    codes, sf = F.mxfp8_quantize(np.zeros((1, 32)))
    assert sf.tolist() == [[127]] and not codes.any()


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def test_mxfp8_golden_block(golden_dir):
    g = _load(golden_dir, "mxfp8_block.json")
    codes, sf = F.mxfp8_quantize(np.array([g["x"]]))
    assert sf.tolist() == [[g["scale_byte"]]]
    assert codes[0].tolist() == g["codes"]


# ----------------------------------------------------------------------------- NVFP4

def test_nvfp4_golden_block(golden_dir):
    g = _load(golden_dir, "nvfp4_block.json")
    x = np.array([g["x"]], dtype=np.float32)
    gs = F.nvfp4_global_scale(np.abs(x).max(1))
    assert np.float32(gs[0]) == np.float32(g["global_scale"])
    packed, sb = F.nvfp4_quantize(x, gs)
    assert sb.tolist() == [[g["block_scale_byte"]]]
    assert F.unpack_e2m1(packed)[0].tolist() == g["codes"]


def test_nvfp4_error_bound():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((32, 256)).astype(np.float32)
    gs = F.nvfp4_global_scale(np.abs(x).max(1))
    packed, sb = F.nvfp4_quantize(x, gs)
    deq = F.nvfp4_dequantize(packed, sb, gs)
    eff = F.E4M3_TABLE[sb] * gs[:, None].astype(np.float64)
    q = x.reshape(32, 16, 16) / eff[..., None]
    # where |x/eff| <= 6, the error is at most half an E2M1 step (0.25 below 2, 0.5 to 4, 1 to 6)
    step = np.where(np.abs(q) < 2, 0.5, np.where(np.abs(q) < 4, 1.0, 2.0))
    err = np.abs(deq.reshape(32, 16, 16) - x.reshape(32, 16, 16))
    inside = np.abs(q) <= 6 * (1 + 1e-6)
    assert np.all(err[inside] <= 0.5 * step[inside] * eff[..., None].repeat(16, -1)[inside] * (1 + 1e-6))
    # the token's amax block never saturates the E4M3 scale beyond 448
    assert F.E4M3_TABLE[sb].max() <= 448


def test_nvfp4_round_trip_of_exact_grid():
    # a block made of exact E2M1 multiples of its own scale comes back unchanged
    gs = np.float32(1.0 / 8)
    sbv = 4.0                                          # E4M3 0x48
    eff = sbv * float(gs)
    codes = np.arange(16, dtype=np.uint8)             # holds +-6, so amax = 6 * eff
    x = (F.E2M1_TABLE[codes] * eff).astype(np.float32)[None]
    # amax/(gs*6) = 4.0 exactly -> sb 0x48 -> the same eff -> the same codes
    packed, sb = F.nvfp4_quantize(x, gs)
    assert sb.tolist() == [[0x48]]
    assert np.array_equal(F.unpack_e2m1(packed)[0] & 0x7, codes & 0x7)
    assert np.array_equal(F.nvfp4_dequantize(packed, sb, gs)[0], x[0].astype(np.float64))


def test_nvfp4_zero_token():
    gs = F.nvfp4_global_scale(np.zeros(1, np.float32))
    assert gs.tolist() == [1.0]
    packed, sb = F.nvfp4_quantize(np.zeros((1, 16), np.float32), gs)
    assert not packed.any() and not sb.any()


# ----------------------------------------------------------------------------- MXFP4 (E2M1 + UE8M0 per 1x32)

def test_mxfp4_golden_block(golden_dir):
    g = _load(golden_dir, "mxfp4_block.json")
    packed, sf = F.mxfp4_quantize(np.array([g["x"]]))
    assert sf.tolist() == [[g["scale_byte"]]]
    assert packed[0].tolist() == g["packed"]


def test_mxfp4_exponent_exact_powers():
    """amax = 6 * 2^n gives e = n; one ulp above gives n + 1."""
    for n in (-20, -3, -1, 0, 1, 5, 30):
        a = np.ldexp(6.0, n)
        assert int(F.mx_exponent(a, 6.0)) == n
        assert int(F.mx_exponent(np.nextafter(a, np.inf), 6.0)) == n + 1
        assert int(F.mx_exponent(np.nextafter(a, 0.0), 6.0)) == n


def test_mxfp4_round_trip_of_exact_grid():
    """A block of E2M1 values times 2^e whose largest magnitude is 6 * 2^e quantises to
    exactly those codes and scale byte e + 127."""
    rng = np.random.default_rng(7)
    for e in (-10, -1, 0, 3, 12):
        codes = rng.integers(0, 16, size=(4, 32)).astype(np.uint8)
        codes[:, 5] = 7 | (rng.integers(0, 2, size=4) << 3).astype(np.uint8)   # +-6: fixes the exponent
        x = F.E2M1_TABLE[codes] * np.ldexp(1.0, e)
        packed, sf = F.mxfp4_quantize(x)
        assert np.array_equal(sf, np.full((4, 1), e + 127, np.uint8))
        got = F.unpack_e2m1(packed)
        # +0 and -0 both decode to 0; compare values, then signs of the non-zeros
        assert np.array_equal(F.E2M1_TABLE[got], F.E2M1_TABLE[codes])


def test_mxfp4_brute_force_nearest():
    """Codes against an exhaustive nearest-value search over the 8 magnitudes (ties to the
    even code), block by block, on random data including exact midpoints."""
    rng = np.random.default_rng(11)
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    x = rng.normal(size=(64, 32)) * np.exp2(rng.integers(-4, 5, size=(64, 1)))
    x[::7, 3] = np.ldexp(1.25, 2)      # midpoints show up at some scales
    packed, sf = F.mxfp4_quantize(x)
    codes = F.unpack_e2m1(packed)
    for r in range(x.shape[0]):
        e = int(sf[r, 0]) - 127
        assert np.abs(x[r]).max() <= 6.0 * 2.0 ** e and (e == -127 or np.abs(x[r]).max() > 3.0 * 2.0 ** e)
        for i in range(32):
            v = abs(x[r, i]) / 2.0 ** e
            d = np.abs(mags - v)
            best = np.flatnonzero(d == d.min())
            want = best[0] if len(best) == 1 else next(b for b in best if b % 2 == 0)
            assert codes[r, i] & 7 == want, (r, i, v)
            if codes[r, i] & 7:
                assert (codes[r, i] >> 3) == (x[r, i] < 0)


def test_mxfp4_error_bound():
    """|x - dequant(quant(x))| <= half the largest E2M1 gap (1) times the block scale, and
    <= a quarter of the scale where |x| <= the scale (gap 0.5 there)."""
    rng = np.random.default_rng(3)
    x = rng.normal(size=(128, 64)) * 3.0
    packed, sf = F.mxfp4_quantize(x)
    d = F.mxfp4_dequantize(packed, sf)
    scale = np.repeat(np.ldexp(1.0, sf.astype(np.int64) - 127), 32, axis=1)
    err = np.abs(x - d)
    assert np.all(err <= scale * (1 + 1e-12))
    small = np.abs(x) <= scale
    assert np.all(err[small] <= 0.25 * scale[small] * (1 + 1e-12))


def test_mxfp4_zero_block():
    packed, sf = F.mxfp4_quantize(np.zeros((2, 32)))
    assert np.all(packed == 0) and np.all(sf == 127)
