"""Pins of the oracle's Q4_K decoding and encoding (the 4-bit sibling format of routed experts).

Format reading: the GGUF Q4_K layout, which the pages keep (QuarkStar (q36) README,
"Acknowledgements"; Q4_K experts in its "Model Weights" section).  The checks tie the
oracle to something other than itself: blocks built byte by byte with hand-derived values
(tests/golden/q4k_blocks.json), nibble probes placed here byte by byte, a pack/unpack round
trip over every field value, the dequantisation formula evaluated here on random fields,
the encoder's error bound derived from its rounding rule, and the whole layer with Q4_K
experts against a dense dequantise-then-matmul brute force.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import qs_inputs as qi

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q4k_blocks.json")


def _block(d_hex, dmin_hex, scales_hex, qs_fill, qs_set=None):
    b = np.zeros(144, np.uint8)
    b[0:2] = np.frombuffer(bytes.fromhex(d_hex), np.uint8)
    b[2:4] = np.frombuffer(bytes.fromhex(dmin_hex), np.uint8)
    b[4:16] = np.frombuffer(bytes.fromhex(scales_hex), np.uint8)
    b[16:144] = qs_fill
    for idx, v in (qs_set or {}).items():
        b[16 + int(idx)] = v
    return b


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)["blocks"]


@pytest.mark.parametrize("blk", _golden(), ids=lambda b: b["name"])
def test_golden_blocks(blk):
    b = _block(blk["d"], blk["dmin"], blk["scales"], blk["qs_fill"], blk.get("qs_set"))
    w = oracle.q4k_dequant(b, 1, 256)[0]
    if "expect_sub" in blk:
        exp = np.repeat(np.array(blk["expect_sub"], np.float64), 32)
    else:
        exp = np.full(256, blk.get("expect_all", 0.0))
        for i, v in blk.get("expect_at", {}).items():
            exp[int(i)] = v
    assert np.array_equal(w, exp)
    if "expect_sc" in blk:
        sc, m, _, _, _ = oracle.q4k_unpack(b)
        assert list(sc) == blk["expect_sc"] and list(m) == blk["expect_m"]


@pytest.mark.parametrize("c", [0, 1, 2, 3])
@pytest.mark.parametrize("high", [False, True])
def test_nibble_probes_fix_the_code_order(c, high):
    # one code of 7 at byte qs[32c + 9]: weight 64c + 9 (low nibble) or 64c + 41 (high nibble)
    b = _block("003c", "0000", "010101010000000001010101", 0, {str(32 * c + 9): (7 << 4) if high else 7})
    w = oracle.q4k_dequant(b, 1, 256)[0]
    exp = np.zeros(256)
    exp[64 * c + 9 + (32 if high else 0)] = 7.0
    assert np.array_equal(w, exp)


@pytest.mark.parametrize("j", range(8))
def test_each_scale_and_min_reaches_only_its_sub_block(j):
    rng = np.random.default_rng(100 + j)
    sc = np.zeros(8, np.uint8)
    m = np.zeros(8, np.uint8)
    sc[j], m[j] = 37, 51          # both above 15: the high bits live in another byte
    q = rng.integers(0, 16, 256).astype(np.uint8)
    b = oracle.q4k_pack(sc, m, q, 0x3C00, 0x3800)   # d = 1, dmin = 0.5
    w = oracle.q4k_dequant(b, 1, 256)[0]
    seg = slice(32 * j, 32 * j + 32)
    assert np.array_equal(w[seg], 37.0 * q[seg] - 25.5)
    rest = np.ones(256, bool)
    rest[seg] = False
    assert np.all(w[rest] == 0.0)


def test_pack_unpack_roundtrip():
    rng = np.random.default_rng(3)
    for _ in range(200):
        sc = rng.integers(0, 64, 8).astype(np.uint8)
        m = rng.integers(0, 64, 8).astype(np.uint8)
        q = rng.integers(0, 16, 256).astype(np.uint8)
        d, dm = int(rng.integers(0, 1 << 16)), int(rng.integers(0, 1 << 16))
        b = oracle.q4k_pack(sc, m, q, d, dm)
        sc2, m2, q2, d2, dm2 = oracle.q4k_unpack(b)
        assert np.array_equal(sc, sc2) and np.array_equal(m, m2) and np.array_equal(q, q2)
        assert (d, dm) == (d2, dm2)


def test_dequant_is_the_formula_on_random_fields():
    rng = np.random.default_rng(4)
    rows = []
    exp = []
    for _ in range(6):
        sc = rng.integers(0, 64, 8).astype(np.uint8)
        m = rng.integers(0, 64, 8).astype(np.uint8)
        q = rng.integers(0, 16, 256).astype(np.uint8)
        d = np.float16(rng.uniform(-1e-2, 1e-2))
        dm = np.float16(rng.uniform(-1e-2, 1e-2))
        rows.append(oracle.q4k_pack(sc, m, q, int(d.view(np.uint16)), int(dm.view(np.uint16))))
        j = np.arange(256) // 32
        exp.append(float(d) * sc[j].astype(np.float64) * q - float(dm) * m[j].astype(np.float64))
    w = oracle.q4k_dequant(np.concatenate(rows), 3, 512)   # rows of two consecutive blocks
    assert np.array_equal(w.reshape(-1), np.concatenate(exp))


def test_quantizer_fixed_point_on_representable_block():
    # d = 2^-10 and dmin = 2^-11 are exact in fp16; one sub-block has scale 63 and one has min 63,
    # so d = max(s)/63 and dmin = max(m)/63 come back exactly; every sub-block uses codes 0 and
    # 15, so its min is -dmin*mc and its max + min is 15*d*sc.  All values are short dyadic
    # numbers, exact in fp32, and re-encoding must give the same bytes.
    rng = np.random.default_rng(8)
    sc = np.array([63, 1, 17, 40, 5, 33, 62, 9], np.uint8)
    m = np.array([0, 63, 12, 1, 48, 7, 30, 21], np.uint8)
    q = rng.integers(0, 16, 256).astype(np.uint8)
    for j in range(8):
        q[32 * j] = 0
        q[32 * j + 31] = 15
    b = oracle.q4k_pack(sc, m, q, 0x1400, 0x1000)   # fp16 bits of 2^-10 and 2^-11
    w = oracle.q4k_dequant(b, 1, 256)
    assert np.array_equal(w.astype(np.float32).astype(np.float64), w)
    again = oracle.q4k_quantize(w.astype(np.float32))
    assert np.array_equal(again.reshape(-1), b)


def test_quantizer_fixed_point_with_an_all_positive_sub_block():
    # The encoder's min is m = max(0, -min w).  Sub-block 3 has min 0 and codes 1..15 only, so
    # all its weights are positive: its m must be 0 and its step max/15 (an unclamped min would
    # give the step (max - min)/15 and the scale 37 in place of 40).  Scale 63 and min 63 fix d
    # and dmin as in the fixed point above; the other sub-blocks use codes 0 and 15.
    rng = np.random.default_rng(10)
    sc = np.array([63, 1, 17, 40, 5, 33, 62, 9], np.uint8)
    m = np.array([5, 63, 12, 0, 48, 7, 30, 21], np.uint8)
    q = rng.integers(0, 16, 256).astype(np.uint8)
    for j in range(8):
        q[32 * j], q[32 * j + 31] = 0, 15
    q[96:128] = rng.integers(1, 16, 32)
    q[96], q[127] = 1, 15
    b = oracle.q4k_pack(sc, m, q, 0x1400, 0x1000)   # d = 2^-10, dmin = 2^-11
    w = oracle.q4k_dequant(b, 1, 256)
    assert np.all(w[0, 96:128] > 0)
    assert np.array_equal(w.astype(np.float32).astype(np.float64), w)
    assert np.array_equal(oracle.q4k_quantize(w.astype(np.float32)).reshape(-1), b)


def test_quantizer_zero_row_gives_zero_block():
    q = oracle.q4k_quantize(np.zeros((1, 256), np.float32))
    assert np.all(oracle.q4k_dequant(q, 1, 256) == 0.0)


def test_quantizer_error_bound_on_gaussian_rows():
    # per sub-block the grid is -dmin*mc + k*d*sc (k = 0..15); rounding to the nearest grid
    # point errs by at most half a step inside the grid; the grid ends miss [min, max] by at
    # most dmin/2 (min code rounding) + 15*d/2 (scale code rounding) + fp16 rounding of d, dmin
    rng = np.random.default_rng(6)
    w = (rng.standard_normal((64, 1024)) * 0.02).astype(np.float32)
    q = oracle.q4k_quantize(w)
    wq = oracle.q4k_dequant(q, 64, 1024)
    for r in range(64):
        for b in range(4):
            sc, m, codes, dh, mh = oracle.q4k_unpack(q[r, b * 144:(b + 1) * 144])
            assert codes.max() <= 15 and sc.max() <= 63 and m.max() <= 63
            d = float(np.uint16(dh).view(np.float16))
            dm = float(np.uint16(mh).view(np.float16))
            for j in range(8):
                seg = slice(b * 256 + 32 * j, b * 256 + 32 * j + 32)
                err = np.abs(wq[r, seg] - w[r, seg].astype(np.float64)).max()
                bound = 0.5 * d * sc[j] + 0.5 * dm + 7.5 * d + 2e-3 * (d * 63 + dm * 63) + 1e-9
                assert err <= bound, (r, b, j, err, bound)
    rel = np.sqrt(np.mean((wq - w) ** 2) / np.mean(w.astype(np.float64) ** 2))
    assert rel < 0.12   # 4-bit codes: far finer than the 2-bit format


def _silu(z):
    return z / (1.0 + np.exp(-z))


def _mlp(Wg, Wu, Wd, x):
    return Wd @ (_silu(Wg @ x) * (Wu @ x))


def test_q4k_layer_against_dense_brute_force():
    shape = qi.LayerShape(512, 8, 2, 256, 256, qi.F32)   # F != H catches a transposed matrix
    E, F, H = shape.n_experts, shape.expert_ffn, shape.hidden
    stride = 144 * 3 * F * H // 256
    experts = np.concatenate([oracle.quantize_expert(*qi.gen_expert_f32(shape, 5, 0, e), fmt="q4k")
                              for e in range(E)])
    assert experts.size == E * stride
    xb, xf = qi.gen_x(shape, 5, 3)
    Wr = qi.gen_router(shape, 5, 0)
    sh = qi.gen_shared(shape, 5, 0)
    out = oracle.moe_ffn(shape, xb, Wr, None, experts, stride, sh, fmt="q4k")
    gb = F * H // 256 * 144

    def dense(e):
        blob = experts[e * stride:(e + 1) * stride]
        return (oracle.q4k_dequant(blob[:gb], F, H), oracle.q4k_dequant(blob[gb:2 * gb], F, H),
                oracle.q4k_dequant(blob[2 * gb:], H, F))

    Sg, Su, Sd = (qi.bf16_bits_to_f32(sh[n]).astype(np.float64) for n in ("gate", "up", "down"))
    ssig = qi.bf16_bits_to_f32(sh["sig"]).astype(np.float64)
    for t in range(3):
        x = xf[t].astype(np.float64)
        l = Wr.astype(np.float64) @ x
        top = sorted(range(E), key=lambda e: (-l[e], e))[:shape.top_k]
        w = np.exp(l[top] - l[top].max())
        w /= w.sum()
        ref = sum(w[j] * _mlp(*dense(e), x) for j, e in enumerate(top))
        ref = ref + _mlp(Sg, Su, Sd, x) / (1.0 + math.exp(-(ssig @ x)))
        assert list(out["ids"][t]) == top
        assert np.allclose(out["y"][t], ref, rtol=1e-10, atol=1e-13)


def test_q2k_is_still_the_default_format():
    shape = qi.WORKLOADS["tiny"].shape
    experts = np.concatenate([oracle.quantize_expert(*qi.gen_expert_f32(shape, 0, 0, e))
                              for e in range(shape.n_experts)])
    xb, _ = qi.gen_x(shape, 0, 2)
    Wr = qi.gen_router(shape, 0, 0)
    a = oracle.moe_ffn(shape, xb, Wr, None, experts, shape.expert_bytes, None)
    b = oracle.moe_ffn(shape, xb, Wr, None, experts, shape.expert_bytes, None, fmt="q2k")
    assert np.array_equal(a["y"], b["y"])
