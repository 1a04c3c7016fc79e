"""The seeded generator is deterministic, counter-based and close to N(0,1)."""
import numpy as np

import csa2_synth as S


def test_counter_based_slices_agree():
    k = S.stream_key(1236, S.S_ENTRIES, 3)
    full = S.normal_f32(k, 0, 5000)
    assert np.array_equal(full[1234:2000], S.normal_f32(k, 1234, 766))
    assert np.array_equal(full, S.normal_f32(k, 0, 5000, chunk=333))


def test_streams_differ_and_repeat():
    a = S.normal_f32(S.stream_key(1, S.S_Q, 0), 0, 100)
    b = S.normal_f32(S.stream_key(1, S.S_Q, 1), 0, 100)
    c = S.normal_f32(S.stream_key(2, S.S_Q, 0), 0, 100)
    assert not np.array_equal(a, b) and not np.array_equal(a, c)
    assert np.array_equal(a, S.normal_f32(S.stream_key(1, S.S_Q, 0), 0, 100))


def test_moments_and_support():
    z = S.normal_f32(S.stream_key(7, S.S_ENTRIES, 0), 0, 1 << 20).astype(np.float64)
    assert abs(z.mean()) < 5e-3 and abs(z.var() - 1.0) < 5e-3
    assert np.abs(z).max() <= 6.0
    kurt = ((z - z.mean()) ** 4).mean() / z.var() ** 2
    assert abs(kurt - 3.0) < 0.15           # Irwin-Hall(12): 3 - 0.1


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.005859375, 1.0078125, -2.5, 3.0e38], np.float32)
    got = S.f32_to_bf16_bits(x)
    assert list(got) == [0x3F80, 0x3F80, 0x3F81, 0x3F81, 0xC020, 0x7F62]


def test_lengths_and_channels():
    L = S.seq_lengths(1237, 4, 524288, 1048576)
    assert np.all((L >= 524288) & (L <= 1048576))
    ch = S.choose_channels(1236, 512, 5)
    assert len(set(ch.tolist())) == 5 and np.all((ch >= 0) & (ch < 512))
