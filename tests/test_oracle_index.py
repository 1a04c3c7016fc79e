"""Pins of the oracle's index score and top-k (blog reading of the DeepSeek-V4
report, section 4.1: I[t,s] = sum_h w[t,h] ReLU(q[t,h] . K[s]); top-k per
query, k = 512 in the V4.1 report, section 4.2.1)."""
import numpy as np
import pytest

import oracle as O
from csa2_synth import bf16_bits_to_f32, f32_to_bf16_bits


def _bf(rng, shape):
    return f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32))


def test_scores_brute_force_tiny():
    rng = np.random.default_rng(0)
    k, q = _bf(rng, (7, 5)), _bf(rng, (3, 5))
    w = rng.standard_normal(3).astype(np.float32)
    got = O.index_scores(k, q, w)
    kf, qf = bf16_bits_to_f32(k).tolist(), bf16_bits_to_f32(q).tolist()
    for s in range(7):
        tot = 0.0
        for h in range(3):
            dot = sum(float(a) * float(b) for a, b in zip(qf[h], kf[s]))
            tot += float(w[h]) * max(dot, 0.0)
        assert got[s] == pytest.approx(tot, rel=1e-12, abs=1e-12)


def test_zero_query_scores_zero_and_selects_first_k():
    rng = np.random.default_rng(1)
    k = _bf(rng, (2048, 128))
    q = np.zeros((32, 128), np.uint16)
    w = rng.standard_normal(32).astype(np.float32)
    idx, sc = O.index_topk(k, q, w, 512)
    assert np.all(sc == 0.0)
    assert np.array_equal(idx, np.arange(512))


def test_single_positive_head_reduces_to_relu_dot():
    rng = np.random.default_rng(2)
    k, q = _bf(rng, (300, 128)), _bf(rng, (32, 128))
    w = np.zeros(32, np.float32)
    w[7] = 1.0
    sc = O.index_scores(k, q, w)
    dots = bf16_bits_to_f32(k).astype(np.float64) @ bf16_bits_to_f32(q[7]).astype(np.float64)
    assert np.allclose(sc, np.maximum(dots, 0.0), rtol=1e-12, atol=1e-9)
    assert np.any(dots < 0) and np.all(sc[dots < 0] == 0.0)


def test_scores_are_linear_in_head_weights():
    rng = np.random.default_rng(3)
    k, q = _bf(rng, (200, 16)), _bf(rng, (4, 16))
    w1 = rng.standard_normal(4).astype(np.float32)
    w2 = rng.standard_normal(4).astype(np.float32)
    a = O.index_scores(k, q, w1) + O.index_scores(k, q, w2)
    b = O.index_scores(k, q, (w1.astype(np.float64) + w2).astype(np.float32))
    assert np.allclose(a, b, rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("n", [0, 1, 5, 511, 512, 513, 3000])
def test_topk_brute_force(n):
    rng = np.random.default_rng(n)
    s = rng.integers(-20, 20, n).astype(np.float32)        # many exact ties
    got = O.topk(s, 512)
    order = sorted(range(n), key=lambda i: (-float(s[i]), i))
    want = sorted(order[:min(512, n)]) + [-1] * (512 - min(512, n))
    assert list(got) == want


def test_topk_all_ties_take_lowest_indices():
    s = np.full(4096, 1.5, np.float32)
    assert np.array_equal(O.topk(s, 512), np.arange(512))


def test_topk_planted_tie_at_the_boundary():
    s = np.zeros(1000, np.float32)
    s[:510] = 10.0                 # 510 clear winners
    s[[700, 600, 900, 650]] = 5.0  # four candidates for the last two slots
    got = O.topk(s, 512)
    assert list(got) == list(range(510)) + [600, 650]


def test_topk_handles_negative_and_signed_zero():
    s = np.array([-0.0, 0.0, -1.0, -1e-30, 1e-30], np.float32)
    got = O.topk(s, 3)
    assert list(got) == [0, 1, 4]          # -0 == +0, lower index first
