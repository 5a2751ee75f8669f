"""Pins of the oracle's directional steering, y <- y - scale * d * (d . y) per row.

Definition: QuarkStar (q36) README, "Steering" (the DwarfStar (ds4) page's
"Steering" section uses the same projection).  The pins are hand-worked rows
(tests/golden/steer_cases.json) and closed-form properties of the projection:
a unit direction with scale 1 leaves nothing along d, twice is the same as
once, scale 2 is a reflection, the part orthogonal to d never changes, and
the edit is linear in y.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "steer_cases.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_hand_worked_rows(case):
    got = oracle.steer_rows(np.array(case["y"]), np.array(case["d"], np.float32), case["scale"])
    assert np.array_equal(got, np.array(case["expect"], np.float64))


def _unit(rng, H):
    d = rng.standard_normal(H)
    return (d / np.linalg.norm(d)).astype(np.float32)


def _rows(rng, T, H):
    return rng.standard_normal((T, H))


def test_unit_direction_removed():
    rng = np.random.default_rng(11)
    d = _unit(rng, 2048)
    y = _rows(rng, 5, 2048)
    out = oracle.steer_rows(y, d, 1.0)
    dd = d.astype(np.float64)
    nd = float(dd @ dd)  # 1 up to the fp32 rounding of d
    # what is left along d is (1 - d.d) times what was there
    for t in range(5):
        assert abs(dd @ out[t] - (1.0 - nd) * (dd @ y[t])) <= 1e-12 * np.linalg.norm(y[t])


def test_projection_is_idempotent():
    rng = np.random.default_rng(12)
    d = np.zeros(64, np.float32)
    d[[3, 17, 40, 63]] = 0.5  # exactly unit length
    y = _rows(rng, 3, 64)
    once = oracle.steer_rows(y, d, 1.0)
    twice = oracle.steer_rows(once, d, 1.0)
    assert np.allclose(twice, once, rtol=0, atol=1e-14)


def test_scale_two_reflects():
    rng = np.random.default_rng(13)
    d = np.zeros(256, np.float32)
    d[::16] = 0.25  # 16 entries of 1/4: exactly unit length
    y = _rows(rng, 4, 256)
    out = oracle.steer_rows(y, d, 2.0)
    dd = d.astype(np.float64)
    for t in range(4):
        assert abs(dd @ out[t] + dd @ y[t]) <= 1e-12 * np.linalg.norm(y[t])
        assert abs(np.linalg.norm(out[t]) - np.linalg.norm(y[t])) <= 1e-12 * np.linalg.norm(y[t])


def test_orthogonal_part_unchanged():
    rng = np.random.default_rng(14)
    H = 512
    d = _unit(rng, H)
    y = _rows(rng, 3, H)
    out = oracle.steer_rows(y, d, 0.8)
    dd = d.astype(np.float64)
    dd = dd / np.linalg.norm(dd)
    perp_in = y - np.outer(y @ dd, dd)
    perp_out = out - np.outer(out @ dd, dd)
    assert np.allclose(perp_out, perp_in, rtol=0, atol=1e-12)
    # and only the component along d moved, by scale * (d . y) * |d|^2
    d64 = d.astype(np.float64)
    moved = (y - out) @ dd
    assert np.allclose(moved, 0.8 * (y @ d64) * np.linalg.norm(d64), rtol=1e-12, atol=1e-12)


def test_linear_in_y():
    rng = np.random.default_rng(15)
    d = _unit(rng, 128)
    y1, y2 = _rows(rng, 2, 128), _rows(rng, 2, 128)
    lhs = oracle.steer_rows(2.0 * y1 - 3.0 * y2, d, -0.7)
    rhs = 2.0 * oracle.steer_rows(y1, d, -0.7) - 3.0 * oracle.steer_rows(y2, d, -0.7)
    assert np.allclose(lhs, rhs, rtol=0, atol=1e-12)


def test_rows_are_independent():
    rng = np.random.default_rng(16)
    d = _unit(rng, 96)
    y = _rows(rng, 6, 96)
    whole = oracle.steer_rows(y, d, 0.3)
    for t in range(6):
        assert np.array_equal(whole[t], oracle.steer_rows(y[t:t + 1], d, 0.3)[0])


def test_length_mismatch_rejected():
    with pytest.raises(ValueError):
        oracle.steer_rows(np.zeros((1, 8)), np.zeros(7, np.float32), 1.0)
