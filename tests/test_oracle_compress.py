"""Pins of the oracle's exp and CSA2 compressor ("DeepSeek-V4.1-Flash"
report, section 2.3: non-overlapping blocks of m tokens, no positional bias;
neshdevtech article section 3.3.2: the gated pooling degenerates to a
per-token projection at m = 1)."""
import math

import numpy as np
import pytest

import oracle as O
from csa2_synth import bf16_bits_to_f32, f32_to_bf16_bits


def _ulp_dist(a, b):
    ia = np.float32(a).view(np.int32).astype(np.int64)
    ib = np.float32(b).view(np.int32).astype(np.int64)
    return abs(int(ia) - int(ib))


def test_exp_within_two_ulp_of_libm():
    rng = np.random.default_rng(0)
    xs = np.concatenate([np.linspace(-87, 0, 30001, dtype=np.float32),
                         rng.uniform(-87, 0, 20000).astype(np.float32),
                         np.float32([-1e-7, -1e-30, -0.0, 0.0])])
    worst = max(_ulp_dist(O.expf(float(x)), math.exp(float(x))) for x in xs)
    assert worst <= 2
    assert O.expf(0.0) == 1.0
    assert O.expf(-90.0) == 0.0
    ys = [O.expf(float(x)) for x in np.linspace(-20, 0, 5001, dtype=np.float32)]
    assert all(b >= a for a, b in zip(ys, ys[1:]))


def test_exp_coefficients_are_rounded_reciprocal_factorials():
    # the device twin spells these as hex literals; they must be RN(1/k!)
    for k in range(2, 8):
        assert np.float32(1.0) / np.float32(math.factorial(k)) == \
            np.float32(1.0 / math.factorial(k))


def _tokens(rng, t, dim=512):
    c = f32_to_bf16_bits(rng.standard_normal((t, dim)).astype(np.float32))
    z = rng.standard_normal((t, dim)).astype(np.float32)
    return c, z


def test_m1_is_bitwise_identity():
    rng = np.random.default_rng(1)
    c, z = _tokens(rng, 64)
    c[0, :4] = [0x8000, 0x0001, 0x8001, 0x7F7F]     # -0, subnormals, max finite
    out = O.compress(c, z, 1)
    assert np.array_equal(out.view(np.uint32), bf16_bits_to_f32(c).view(np.uint32))


@pytest.mark.parametrize("m", [2, 4, 8])
def test_equal_logits_give_the_exact_mean(m):
    rng = np.random.default_rng(m)
    c, _ = _tokens(rng, 32 * m)
    z = np.repeat(rng.standard_normal((32, 512)).astype(np.float32), m, axis=0)
    out = O.compress(c, z, m)
    cf = bf16_bits_to_f32(c).reshape(32, m, 512)
    acc = cf[:, 0].copy()
    for j in range(1, m):
        acc = (acc + cf[:, j]).astype(np.float32)
    assert np.array_equal(out, (acc * np.float32(1.0 / m)).astype(np.float32))


def test_dominant_logit_selects_its_token():
    rng = np.random.default_rng(3)
    c, z = _tokens(rng, 64)
    z[0::2] = 50.0
    z[1::2] = -50.0          # difference 100 > 87: the other weight is exactly 0
    out = O.compress(c, z, 2)
    assert np.array_equal(out, bf16_bits_to_f32(c[0::2]))


def test_matches_fp64_softmax_pooling():
    rng = np.random.default_rng(4)
    for m in (2, 3, 4):
        c, z = _tokens(rng, 40 * m)
        z *= 3.0
        out = O.compress(c, z, m).astype(np.float64)
        cf = bf16_bits_to_f32(c).astype(np.float64).reshape(40, m, 512)
        zz = z.astype(np.float64).reshape(40, m, 512)
        w = np.exp(zz - zz.max(axis=1, keepdims=True))
        w /= w.sum(axis=1, keepdims=True)
        ref = (w * cf).sum(axis=1)
        scale = np.abs(cf).max(axis=1)
        assert np.all(np.abs(out - ref) <= 8 * 2.0 ** -24 * m * scale + 1e-30)
        # a convex combination per channel
        assert np.all(out <= cf.max(axis=1) + 1e-6) and np.all(out >= cf.min(axis=1) - 1e-6)


def test_channels_are_independent():
    rng = np.random.default_rng(6)
    c, z = _tokens(rng, 16)
    perm = rng.permutation(512)
    a = O.compress(c, z, 2)[:, perm]
    b = O.compress(c[:, perm], z[:, perm], 2)
    assert np.array_equal(a, b)
