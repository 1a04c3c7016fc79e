"""Pins of the oracle's FP8 window rows ("DeepSeek-V4.1-Flash" report,
section 2.4.4: the SWA KV cache stays FP8; the V4 FP8 row: 448 FP8 + 64
bf16 RoPE channels + 8 bytes of scale = 584 bytes)."""
import numpy as np
import pytest

import oracle as O
from csa2_synth import f32_to_bf16_bits, bf16_bits_to_f32
from tests._golden import numbers

G = numbers()


def _rows(rng, n, spread=6):
    x = rng.standard_normal((n, 512)) * np.exp(rng.uniform(-spread, spread, (n, 1)))
    return f32_to_bf16_bits(x.astype(np.float32))


def test_row_bytes():
    rng = np.random.default_rng(0)
    c, r, s = O.swa_fp8_quantise(_rows(rng, 3))
    assert c.shape[1] + 2 * r.shape[1] + s.shape[1] == G["v4_main_entry_bytes"] == 584


def test_codes_match_the_library_conversion():
    """The per-64-channel scale is the OCP MX one (floor(log2 amax) - 8); the
    codes of x / scale are torch's float32 -> float8_e4m3fn conversion
    (nearest even) wherever the quotient stays within 448."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    x = _rows(rng, 64)
    codes, rope, scales = O.swa_fp8_quantise(x)
    xf = bf16_bits_to_f32(x).astype(np.float64)
    for blk in range(7):
        xb = xf[:, 64 * blk:64 * blk + 64]
        amax = np.abs(xb).max(axis=1)
        want = np.floor(np.log2(amax)).astype(int) - 8 + 127
        assert np.array_equal(scales[:, blk], want)
        q = (xb / 2.0 ** (want[:, None] - 127)).astype(np.float32)
        ok = np.abs(q) <= 448
        ref = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(codes[:, 64 * blk:64 * blk + 64][ok], ref[ok])
        assert np.all(codes[:, 64 * blk:64 * blk + 64][~ok] & 0x7F == 0x7E)   # saturated
    assert np.all(scales[:, 7] == 0)
    assert np.array_equal(rope, x[:, 448:])


def test_round_trip_error_bound_and_fixed_points():
    rng = np.random.default_rng(2)
    x = _rows(rng, 50)
    r = O.swa_fp8_round_bf16(x)
    assert np.array_equal(O.swa_fp8_round_bf16(r), r)             # idempotent
    assert np.array_equal(r[:, 448:], x[:, 448:])                 # RoPE channels exact
    xf = bf16_bits_to_f32(x).astype(np.float64)
    rf = bf16_bits_to_f32(r).astype(np.float64)
    _, _, scales = O.swa_fp8_quantise(x)
    for blk in range(7):
        s = 2.0 ** (scales[:, blk].astype(np.float64) - 127)[:, None]
        a = np.abs(xf[:, 64 * blk:64 * blk + 64]) / s
        # E4M3 step at a: 2^(floor(log2 a) - 3) for normals, 2^-9 below 2^-6
        step = np.where(a >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(a, 1e-30))) - 3), 2.0 ** -9)
        bound = np.where(a > 448, (a - 448) * s, step / 2 * s)
        err = np.abs(xf[:, 64 * blk:64 * blk + 64] - rf[:, 64 * blk:64 * blk + 64])
        assert np.all(err <= bound * (1 + 1e-12))


def test_zero_and_tiny_blocks():
    x = np.zeros((2, 512), np.uint16)
    x[1, 5] = f32_to_bf16_bits(np.array([1e-30], np.float32))[0]
    codes, rope, scales = O.swa_fp8_quantise(x)
    assert np.all(codes[0] == 0) and np.all(scales[0] == 0)
    r = O.swa_fp8_round_bf16(x)
    assert np.all(r[0] == 0)
