"""Pins of the oracle's MXFP4 indexer ("DeepSeek-V4.1-Flash" report, section
2.4.4: FP4 indexer queries and keys in OCP MXFP4; 68 B per key)."""
import numpy as np

import oracle as O
from csa2_synth import f32_to_bf16_bits, bf16_bits_to_f32
from tests._golden import numbers

G = numbers()


def test_key_bytes():
    # 64 bytes of E2M1 codes + 4 UE8M0 scales per 128 channels
    assert O.entry_bytes(128, O.LAYOUT_L32_UE8M0) == 68


def test_grid_rounding_is_idempotent_and_exact_on_grid_values():
    rng = np.random.default_rng(0)
    x = f32_to_bf16_bits((rng.standard_normal((50, 128)) * np.exp(rng.uniform(-8, 8, (50, 1))))
                         .astype(np.float32))
    r = O.mxfp4_round_bf16(x)
    assert np.array_equal(O.mxfp4_round_bf16(r), r)
    # a block of E2M1 values times 2^e is already on the grid
    codes = rng.integers(0, 16, (7, 128))
    vals = np.array([O.e2m1_value(int(c)) for c in codes.ravel()], np.float32).reshape(7, 128)
    vals[:, ::32] = 6.0                      # amax 6 in every block: scale 1
    g = f32_to_bf16_bits(vals * np.float32(2.0 ** -3))
    assert np.array_equal(O.mxfp4_round_bf16(g), g)


def test_rounding_error_within_half_a_step():
    """With the block scale s = 2^(floor(log2 amax) - 2) (OCP MX), |x| / s is
    below 8: up to 6 the error is at most half the E2M1 step times s, above
    6 the value clips to 6 s."""
    rng = np.random.default_rng(1)
    x = f32_to_bf16_bits(rng.standard_normal((40, 128)).astype(np.float32))
    xf = bf16_bits_to_f32(x).astype(np.float64).reshape(-1, 4, 32)
    rf = bf16_bits_to_f32(O.mxfp4_round_bf16(x)).astype(np.float64).reshape(-1, 4, 32)
    amax = np.abs(xf).max(axis=2, keepdims=True)
    s = 2.0 ** (np.floor(np.log2(amax)) - 2)
    a = np.abs(xf) / s
    assert np.all(a < 8)
    step = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    bound = np.where(a > 6, (a - 6) * s, step / 2 * s)
    assert np.all(np.abs(xf - rf) <= bound + 1e-12)
    clipped = a > 6
    assert clipped.any() and np.all(np.abs(rf[clipped]) == 6 * np.broadcast_to(s, a.shape)[clipped])


def test_mxfp4_selection_is_the_bf16_selection_on_rounded_inputs():
    rng = np.random.default_rng(2)
    n = 2500
    k = f32_to_bf16_bits(rng.standard_normal((n, 128)).astype(np.float32))
    q = f32_to_bf16_bits(rng.standard_normal((32, 128)).astype(np.float32))
    w = rng.standard_normal(32).astype(np.float32)
    idx, sc = O.index_topk_mxfp4(k, q, w, 512)
    idx2, sc2 = O.index_topk(O.mxfp4_round_bf16(k), O.mxfp4_round_bf16(q), w, 512)
    assert np.array_equal(idx, idx2) and np.array_equal(sc, sc2)
    # and it is a genuinely different selection from the bf16 one
    full, _ = O.index_topk(k, q, w, 512)
    assert 0.5 < O.recall(idx, full) < 1.0
