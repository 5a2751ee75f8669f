"""Pins of the oracle's Q2_K decoding, encoding and storage conversions.

Every check here ties the oracle to something other than itself: numpy's own
float16 conversion, hand-derived block values (tests/golden/q2k_blocks.json),
single-bit probes built byte by byte in this file, and error bounds derived
from the encoder's rounding rule.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q2k_blocks.json")


# ------------------------------------------------------------------ storage types

def test_half_decode_matches_numpy_for_every_pattern():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(p)) for p in pats])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got) & (got > 0), np.isinf(ref) & (ref > 0))


def test_float_to_half_matches_numpy_rounding():
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(0.05),
        rng.standard_normal(2000).astype(np.float32) * np.float32(3e4),
        (rng.standard_normal(2000) * 1e-6).astype(np.float32),       # subnormal halves
        np.array([65504, 65519.99, 65520, 1e9, 0.0, -0.0, 2.0 ** -25, 2.0 ** -24, 3 * 2.0 ** -26,
                  1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 2049.0, 2051.0], dtype=np.float32),
    ])
    with np.errstate(over="ignore"):  # values past the fp16 range round to infinity on purpose
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.float_to_half(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_decode_is_upper_half_of_fp32():
    rng = np.random.default_rng(1)
    f = rng.standard_normal(1000).astype(np.float32)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ hand-built blocks

def _block(scales_hex, qs_fill, d_hex, dmin_hex, qs_set=None):
    b = np.zeros(84, np.uint8)
    b[0:16] = np.frombuffer(bytes.fromhex(scales_hex), np.uint8)
    b[16:80] = qs_fill
    for idx, v in (qs_set or {}).items():
        b[16 + int(idx)] = v
    b[80:82] = np.frombuffer(bytes.fromhex(d_hex), np.uint8)
    b[82:84] = np.frombuffer(bytes.fromhex(dmin_hex), np.uint8)
    return b


def test_golden_blocks():
    spec = json.load(open(GOLDEN))
    for blk in spec["blocks"]:
        b = _block(blk["scales"], blk["qs_fill"], blk["d"], blk["dmin"], blk.get("qs_set"))
        w = oracle.q2k_dequant(b, 1, 256)[0]
        exp = np.full(256, blk.get("expect_all", 0.0))
        for i, v in blk.get("expect_at", {}).items():
            exp[int(i)] = v
        if "expect_range" in blk:
            r = blk["expect_range"]
            exp[r["start"]:r["stop"]] = r["value"]
        if "expect_pattern_j" in blk:
            j = (np.arange(256) % 128) // 32
            exp = np.array(blk["expect_pattern_j"])[j]
        assert np.array_equal(w, exp), blk["name"]


@pytest.mark.parametrize("h", [0, 1])
@pytest.mark.parametrize("j", [0, 1, 2, 3])
def test_single_bit_probes_fix_the_packing_order(h, j):
    # one code q=1 at byte 32h+l, shift 2j, scale nibble 1, d = 1: exactly weight 128h+32j+l is 1
    for l in (0, 1, 7, 16, 31):
        b = _block("01" * 16, 0, "003c", "0000", {str(32 * h + l): 1 << (2 * j)})
        w = oracle.q2k_dequant(b, 1, 256)[0]
        exp = np.zeros(256)
        exp[128 * h + 32 * j + l] = 1.0
        assert np.array_equal(w, exp)


@pytest.mark.parametrize("s", range(16))
def test_scale_byte_s_covers_weights_16s_to_16s_plus_15(s):
    sc = ["01"] * 16
    sc[s] = "03"
    b = _block("".join(sc), 0x55, "003c", "0000")
    w = oracle.q2k_dequant(b, 1, 256)[0]
    exp = np.ones(256)
    exp[16 * s:16 * s + 16] = 3.0
    assert np.array_equal(w, exp)


def test_rows_are_consecutive_blocks():
    # row of 2 blocks: first all 2.0, second all -1.5
    b0 = _block("11" * 16, 255, "003c", "003c")
    b1 = _block("30" * 16, 255, "003c", "0038")
    w = oracle.q2k_dequant(np.concatenate([b0, b1]), 1, 512)[0]
    assert np.array_equal(w, np.r_[np.full(256, 2.0), np.full(256, -1.5)])


def test_pack_unpack_roundtrip():
    rng = np.random.default_rng(3)
    for _ in range(50):
        sc = rng.integers(0, 256, 16).astype(np.uint8)
        q = rng.integers(0, 4, 256).astype(np.uint8)
        d, m = int(rng.integers(0, 65536)), int(rng.integers(0, 65536))
        blk = oracle.q2k_pack(sc, q, d, m)
        sc2, q2, d2, m2 = oracle.q2k_unpack(blk)
        assert np.array_equal(sc, sc2) and np.array_equal(q, q2) and d == d2 and m == m2


def test_dequant_is_the_formula_on_random_fields():
    rng = np.random.default_rng(4)
    sc = rng.integers(0, 256, 16).astype(np.uint8)
    q = rng.integers(0, 4, 256).astype(np.uint8)
    d = np.float16(0.0123).view(np.uint16)
    m = np.float16(0.0071).view(np.uint16)
    blk = oracle.q2k_pack(sc, q, int(d), int(m))
    w = oracle.q2k_dequant(blk, 1, 256)[0]
    dd = float(np.uint16(d).view(np.float16))
    mm = float(np.uint16(m).view(np.float16))
    s = np.arange(256) // 16
    exp = dd * (sc[s] & 15) * q - mm * (sc[s] >> 4)
    assert np.array_equal(w, exp)


# ------------------------------------------------------------------ encoder

def test_quantizer_fixed_point_on_representable_block():
    # every sub-block holds {-m, -m+s, -m+2s, -m+3s} with s = 15*d0 and m = 15*dm0 exact in fp16:
    # the encoder must find d0, dm0, scale nibbles 15/15 and give the block back exactly
    d0, dm0 = np.float32(np.float16(0.005859375)), np.float32(np.float16(0.001953125))
    s, m = np.float32(15) * d0, np.float32(15) * dm0
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 4, 256)
    for sb in range(16):
        codes[16 * sb:16 * sb + 4] = [0, 1, 2, 3]
    w = (-m + codes.astype(np.float32) * s).astype(np.float32)
    blk = oracle.q2k_quantize(w[None, :])[0]
    sc, q, dh, mh = oracle.q2k_unpack(blk)
    assert dh == np.float16(d0).view(np.uint16) and mh == np.float16(dm0).view(np.uint16)
    assert np.all(sc == 0xFF)
    assert np.array_equal(q, codes)
    assert np.array_equal(oracle.q2k_dequant(blk, 1, 256)[0], w.astype(np.float64))


def test_quantizer_fixed_point_with_an_all_positive_sub_block():
    # The encoder's min is m = max(0, -min w).  Sub-block 5 has min nibble 0 and codes 1..3
    # only, so all its weights are positive: its m must be 0 and its step max/3 (an unclamped
    # min would give the step (max - min)/3 and another scale nibble).  Sub-block 0 carries scale
    # nibble 15 and sub-block 1 min nibble 15, so d and dmin come back exactly; the other
    # sub-blocks use codes 0 and 3, so their min is -dmin*hi and their range is 3*d*lo.
    rng = np.random.default_rng(9)
    lo = np.array([15, 2, 7, 1, 11, 6, 3, 9, 4, 13, 5, 8, 10, 12, 14, 1], np.uint8)
    hi = np.array([0, 15, 3, 9, 1, 0, 7, 2, 11, 4, 13, 6, 8, 5, 10, 12], np.uint8)
    codes = rng.integers(0, 4, 256).astype(np.uint8)
    for sb in range(16):
        codes[16 * sb], codes[16 * sb + 15] = 0, 3
    codes[80:96] = rng.integers(1, 4, 16)
    codes[80], codes[95] = 1, 3
    blk = oracle.q2k_pack(lo | (hi << 4), codes, 0x1400, 0x1000)   # d = 2^-10, dmin = 2^-11
    w = oracle.q2k_dequant(blk, 1, 256)[0]
    assert np.all(w[80:96] > 0)
    assert np.array_equal(w.astype(np.float32).astype(np.float64), w)
    assert np.array_equal(oracle.q2k_quantize(w.astype(np.float32)[None, :])[0], blk)


def test_quantizer_zero_row_gives_zero_block():
    blk = oracle.q2k_quantize(np.zeros((1, 256), np.float32))[0]
    assert np.all(blk == 0)


def test_quantizer_error_bound_on_gaussian_rows():
    # per sub-block the grid is -dmin*hi + k*d*lo (k = 0..3); rounding to the nearest grid point
    # errs by at most half a step inside the grid, and the grid ends miss [min, max] by at most
    # dmin/2 (min nibble rounding) + 3*d/2 (scale nibble rounding) + fp16 rounding of d, dmin.
    rng = np.random.default_rng(6)
    w = (rng.standard_normal((64, 1024)) * 0.02).astype(np.float32)
    q = oracle.q2k_quantize(w)
    wq = oracle.q2k_dequant(q, 64, 1024)
    for r in range(64):
        for b in range(4):
            blk = q[r, b * 84:(b + 1) * 84]
            sc, codes, dh, mh = oracle.q2k_unpack(blk)
            assert codes.max() <= 3
            d = float(np.uint16(dh).view(np.float16))
            dm = float(np.uint16(mh).view(np.float16))
            for sb in range(16):
                lo, hi = sc[sb] & 15, sc[sb] >> 4
                seg = slice(b * 256 + 16 * sb, b * 256 + 16 * sb + 16)
                err = np.abs(wq[r, seg] - w[r, seg].astype(np.float64)).max()
                bound = 0.5 * d * lo + 0.5 * dm + 1.5 * d + 2e-3 * (d * 15 + dm * 15) + 1e-9
                assert err <= bound, (r, b, sb, err, bound)
    rel = np.sqrt(np.mean((wq - w) ** 2) / np.mean(w.astype(np.float64) ** 2))
    assert rel < 0.45   # 2-bit codes: rms error well under half the rms weight
