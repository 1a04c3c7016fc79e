"""Pins of the oracle's readout epilogue variants ("DeepSeek-V4" blog
reading, section 4.3): the attention sink in the softmax denominator and
the output RoPE(-i) on the last 64 channels."""
import numpy as np

import oracle as O
from csa2_synth import f32_to_bf16_bits, bf16_bits_to_f32

SCALE = np.float32(512 ** -0.5)


def _one_query(rng, n_ent=40, n_swa=5, layout=0):
    q = f32_to_bf16_bits(rng.standard_normal((64, 512)).astype(np.float32))
    e = rng.standard_normal((n_ent, 512)).astype(np.float32)
    codes, scales = O.quantise(e, layout)
    swa = f32_to_bf16_bits(rng.standard_normal((n_swa, 512)).astype(np.float32))
    idx = np.arange(n_ent, dtype=np.int32)
    return q, codes, scales, idx, swa


def test_sink_at_minus_infinity_changes_nothing():
    rng = np.random.default_rng(0)
    q, codes, scales, idx, swa = _one_query(rng)
    b, o, l = O.sparse_attention(q, codes, scales, 0, idx, swa, SCALE)
    b2, o2, l2 = O.attention_epilogue(o, l, sink=np.full(64, -np.inf))
    assert np.array_equal(o2, o) and np.array_equal(l2, l) and np.array_equal(b2, b)


def test_sink_with_one_candidate_is_a_sigmoid():
    """One candidate v with logit z against a sink z': the weight is
    e^z / (e^z + e^z') = sigmoid(z - z'), so out = sigmoid(z - z') v."""
    rng = np.random.default_rng(1)
    q, codes, scales, _, _ = _one_query(rng, n_ent=1, n_swa=0)
    _, o, l = O.sparse_attention(q, codes, scales, 0, np.array([0], np.int32), None, SCALE)
    v = O.dequantise(codes, scales, 0)[0].astype(np.float64)
    qf = bf16_bits_to_f32(q).astype(np.float64)
    z = float(SCALE) * (qf @ v)
    zs = rng.standard_normal(64) * 3
    _, o2, l2 = O.attention_epilogue(o, l, sink=zs)
    sig = 1.0 / (1.0 + np.exp(zs - z))
    assert np.allclose(o2, sig[:, None] * v[None, :], rtol=1e-12, atol=1e-12)
    assert np.allclose(l2, np.log(np.exp(z) + np.exp(zs)), rtol=0, atol=1e-12)


def test_sink_weights_sum_below_one():
    """With every value equal to 1 the output equals the sum of the weights,
    which the sink pushes below 1 by exactly e^z' / (sum + e^z')."""
    rng = np.random.default_rng(2)
    q = f32_to_bf16_bits(rng.standard_normal((64, 512)).astype(np.float32))
    ones = np.ones((8, 512), np.float32)
    codes, scales = O.quantise(ones, 0)
    _, o, l = O.sparse_attention(q, codes, scales, 0, np.arange(8, dtype=np.int32), None, SCALE)
    assert np.allclose(o, 1.0, atol=1e-12)
    zs = np.linspace(-4, 4, 64)
    _, o2, l2 = O.attention_epilogue(o, l, sink=zs)
    want = 1.0 - np.exp(zs - l2)
    assert np.allclose(o2, want[:, None], atol=1e-12)
    assert np.all(o2 < 1.0)


def test_output_rope_is_a_complex_rotation():
    """Interleaved pairs of the last 64 channels times exp(-i pos theta_t)
    (numpy complex arithmetic); the first 448 channels are untouched;
    position 0 is the identity; rotating back by +pos restores the output."""
    rng = np.random.default_rng(3)
    out = rng.standard_normal((64, 512))
    lse = rng.standard_normal(64)
    for pos in (0, 1, 37, 131071, 1048575):
        _, r, l2 = O.attention_epilogue(out, lse, rope_pos=pos)
        assert np.array_equal(l2, lse)
        assert np.array_equal(r[:, :448], out[:, :448])
        z = out[:, 448::2] + 1j * out[:, 449::2]
        theta = 10000.0 ** (-np.arange(32) / 32.0)
        zr = z * np.exp(-1j * pos * theta)
        assert np.allclose(r[:, 448::2], zr.real, rtol=0, atol=1e-12)
        assert np.allclose(r[:, 449::2], zr.imag, rtol=0, atol=1e-12)
        if pos == 0:
            assert np.array_equal(r, out)
        back = r.copy()
        zb = (back[:, 448::2] + 1j * back[:, 449::2]) * np.exp(1j * pos * theta)
        assert np.allclose(zb, z, atol=1e-9)
        # rotation keeps every pair's norm
        assert np.allclose(np.abs(r[:, 448::2] + 1j * r[:, 449::2]), np.abs(z), atol=1e-12)


def test_sink_and_rope_commute_and_round_to_bf16():
    rng = np.random.default_rng(4)
    out = rng.standard_normal((64, 512))
    lse = rng.standard_normal(64)
    zs = rng.standard_normal(64)
    b1, o1, _ = O.attention_epilogue(out, lse, sink=zs, rope_pos=99)
    _, tmp, l_tmp = O.attention_epilogue(out, lse, rope_pos=99)
    _, o2, _ = O.attention_epilogue(tmp, lse, sink=zs)
    assert np.allclose(o1, o2, atol=1e-14)
    assert np.array_equal(bf16_bits_to_f32(b1), O.bf16_round(o1.astype(np.float32)))


def test_empty_head_without_sink_stays_empty():
    out = np.zeros((64, 512))
    lse = np.full(64, -np.inf)
    zs = np.full(64, 1.5)
    zs[3] = -np.inf
    _, o, l = O.attention_epilogue(out, lse, sink=zs, rope_pos=7)
    assert np.all(o == 0) and np.all(np.isfinite(o))
    assert l[3] == -np.inf and np.all(l[np.arange(64) != 3] == 1.5)
