"""Pins of the oracle's FP4 / FP8 codec against what the pages and the
format definitions fix ("DeepSeek-V4.1-Flash" report, section 2.4.4; OCP
Microscaling Formats v1.0 for E2M1 / E4M3 / UE8M0)."""
import math

import numpy as np
import pytest

import oracle as O
from tests._golden import numbers

G = numbers()
E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_table_is_the_ocp_grid():
    for c in range(8):
        assert O.e2m1_value(c) == E2M1_GRID[c]
        neg = O.e2m1_value(c | 8)
        assert neg == -E2M1_GRID[c] and math.copysign(1.0, neg) == -1.0
    assert max(O.e2m1_value(c) for c in range(16)) == G["e2m1_max"]


def test_e4m3_landmarks():
    assert O.e4m3_value(0x7E) == G["e4m3_max"]
    assert math.isnan(O.e4m3_value(0x7F)) and math.isnan(O.e4m3_value(0xFF))
    assert O.e4m3_value(0x38) == 1.0           # exponent field 7 = bias
    assert O.e4m3_value(0x01) == 2.0 ** -9     # smallest subnormal
    assert O.e4m3_value(0x08) == 2.0 ** -6     # smallest normal
    assert O.e4m3_value(0x07) == 7 * 2.0 ** -9
    vals = [O.e4m3_value(b) for b in range(0x7F)]
    assert all(b > a for a, b in zip(vals, vals[1:]))      # strictly increasing
    assert all(not math.isinf(v) for v in vals)              # no infinities
    assert all(O.e4m3_value(b | 0x80) == -O.e4m3_value(b) for b in range(1, 0x7F))


def test_max_magnitude_is_2688():
    amax = O.e4m3_value(0x7E) * O.e2m1_value(7)
    assert amax == G["fp4_max_magnitude"] == G["e4m3_max"] * G["e2m1_max"]
    # a block whose amax is 2688 keeps it exactly in the E4M3-scale layout
    x = np.zeros((1, 16), np.float32)
    x[0, 3] = 2688.0
    x[0, 5] = -2688.0
    codes, scales = O.quantise(x, O.LAYOUT_L16_E4M3)
    assert scales[0, 0] == 0x7E
    back = O.dequantise(codes, scales, O.LAYOUT_L16_E4M3)
    assert back[0, 3] == 2688.0 and back[0, 5] == -2688.0


@pytest.mark.parametrize("v,code", [
    (0.0, 0), (0.25, 0), (0.2500001, 1), (0.5, 1), (0.75, 2), (1.0, 2), (1.25, 2),
    (1.2500001, 3), (1.5, 3), (1.75, 4), (2.5, 4), (2.5000002, 5), (3.0, 5), (3.5, 6),
    (5.0, 6), (5.0000005, 7), (6.0, 7), (7.0, 7), (1e30, 7), (float("inf"), 7),
    (-0.0, 8), (-0.1, 8), (-0.75, 10), (-5.0, 14), (-100.0, 15)])
def test_e2m1_round_to_nearest_even_saturating(v, code):
    assert O.e2m1_encode(v) == code


def test_e2m1_encode_is_nearest_on_a_dense_sweep():
    xs = np.linspace(-8.0, 8.0, 20001, dtype=np.float32)
    grid = np.array(E2M1_GRID)
    for x in xs[::3]:
        c = O.e2m1_encode(float(x))
        got = O.e2m1_value(c)
        best = np.min(np.abs(abs(float(x)) - grid))
        if abs(x) <= 6.0:
            assert abs(abs(got) - abs(float(x))) == pytest.approx(best, abs=0)
        else:
            assert abs(got) == 6.0


def test_ue8m0_rule_is_ocp_shared_exponent():
    # shared exponent = floor(log2(amax)) - 2  (E2M1 emax = 2)
    assert O.ue8m0_for_amax(6.0) == 127
    assert O.ue8m0_for_amax(4.0) == 127
    assert O.ue8m0_for_amax(7.99) == 127
    assert O.ue8m0_for_amax(8.0) == 128
    assert O.ue8m0_for_amax(1.0) == 125
    assert O.ue8m0_for_amax(0.75) == 124
    assert O.ue8m0_for_amax(0.0) == 0
    assert O.ue8m0_for_amax(1e-45) == 0          # subnormal amax clamps
    assert O.ue8m0_for_amax(3e38) == 127 + 127 - 2
    assert O.ue8m0_value(127) == 1.0 and O.ue8m0_value(0) == 2.0 ** -127
    assert math.isnan(O.ue8m0_value(255))


def test_e4m3_scale_rule():
    assert O.e4m3_encode(1.0) == 0x38
    assert O.e4m3_encode(448.0) == 0x7E and O.e4m3_encode(1e6) == 0x7E
    assert O.e4m3_encode(1.0625) == 0x38          # tie 1.0 / 1.125 -> even code
    assert O.e4m3_encode(1.1875) == 0x3A          # tie 1.125 / 1.25 -> even code
    assert O.e4m3_encode(2.0 ** -10) == 0x00      # half the smallest subnormal -> 0
    assert O.e4m3_encode(3 * 2.0 ** -10) == 0x02  # tie 2^-9 / 2^-8 -> even code
    for b in range(0x7F):
        assert O.e4m3_encode(O.e4m3_value(b)) == b  # every value encodes to itself


@pytest.mark.parametrize("layout", [O.LAYOUT_L32_UE8M0, O.LAYOUT_L16_E4M3])
def test_round_trip_every_code(layout):
    """quant(dequant(code, s)) == code for every code, at many scales: the
    block's amax is pinned to 6 * s so that the rule picks s back."""
    g = O.group(layout)
    if layout == O.LAYOUT_L32_UE8M0:
        scale_bytes = list(range(100, 160))
        svals = [O.ue8m0_value(b) for b in scale_bytes]
    else:
        scale_bytes = [b for b in range(0x08, 0x7F)]
        svals = [O.e4m3_value(b) for b in scale_bytes]
    for sb, s in zip(scale_bytes, svals):
        x = np.zeros((16, g), np.float32)
        x[:, 0] = 6.0 * s
        for c in range(16):
            x[c, 1] = O.e2m1_value(c) * s
        codes, scales = O.quantise(x, layout)
        assert np.all(scales[:, 0] == sb)
        got = codes[:, 0] >> 4          # channel 1 sits in the high nibble
        assert list(got) == list(range(16))


@pytest.mark.parametrize("layout", [O.LAYOUT_L32_UE8M0, O.LAYOUT_L16_E4M3])
def test_error_bound_and_bf16_exactness(layout):
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((4096, 512)) * rng.choice([0.01, 1, 30], (4096, 1))).astype(np.float32)
    codes, scales = O.quantise(x, layout)
    xh = O.dequantise(codes, scales, layout)
    g = O.group(layout)
    s = np.array([[O.ue8m0_value(b) if layout == 0 else O.e4m3_value(b) for b in row]
                  for row in scales[:64]], np.float64)
    s_full = np.repeat(s, g, axis=1)
    err = np.abs(xh[:64].astype(np.float64) - x[:64])
    # half the local E2M1 spacing (0.25 up to 2, 0.5 up to 4, 1 up to 6)
    mag = np.abs(x[:64]) / s_full
    half = np.where(mag <= 2, 0.25, np.where(mag <= 4, 0.5, 1.0))
    inside = mag <= 6
    assert np.all(err[inside] <= half[inside] * s_full[inside])
    # values are e2m1 * scale: at most 2 + 4 significant bits -> exact in bf16
    b = xh.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0)


def test_ue8m0_clips_near_amax_like_ocp():
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 7.5       # amax 7.5 -> s = 1 -> 7.5 saturates to 6
    codes, scales = O.quantise(x, O.LAYOUT_L32_UE8M0)
    assert scales[0, 0] == 127 and (codes[0, 0] & 15) == 7
