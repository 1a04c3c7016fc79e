"""Pins of the oracle's bf16-rounded index scores ("DeepSeek-V4" blog
reading, section 7: scores quantised from FP32 to BF16 before the top-k
selector)."""
import numpy as np
import pytest

import oracle as O


def test_rounding_landmarks():
    one = np.float32(1.0)
    u = np.float32(2.0 ** -7)                      # bf16 spacing in [1, 2)
    cases = [
        (1.0, 1.0),
        (1.0 + 2.0 ** -9, 1.0),                    # below the midpoint
        (1.0 + 2.0 ** -8, 1.0),                    # midpoint, 1.0 is even
        (1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -6),    # midpoint, 1 + 2^-6 is even
        (1.0 + 2.0 ** -8 + 2.0 ** -20, 1.0 + 2.0 ** -7),
        (-(1.0 + 2.0 ** -8), -1.0),
        (3.140625, 3.140625),                      # already a bf16 value
        (0.0, 0.0),
    ]
    for x, want in cases:
        assert O.bf16_round(np.float32(x)) == np.float32(want), x
    assert np.signbit(O.bf16_round(np.float32(-0.0)))
    assert one + u == O.bf16_round(one + u)


def test_matches_the_library_conversion():
    """Against torch's float32 -> bfloat16 conversion (round to nearest
    even), on random values and on every exact midpoint of a sample."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-30, 30, 200000))).astype(np.float32)
    bits = x.view(np.uint32)
    mids = ((bits & 0xFFFF0000) | 0x8000).astype(np.uint32).view(np.float32)
    for v in (x, mids):
        ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
        assert np.array_equal(O.bf16_round(v), ref)


def test_rounding_creates_ties_that_go_to_the_lower_index():
    s = np.array([1.0, 1.0 + 2.0 ** -9, 0.5, 1.0 + 2.0 ** -10, 2.0], np.float32)
    b = O.bf16_round(s)
    assert list(b) == [1.0, 1.0, 0.5, 1.0, 2.0]
    # fp32 order would pick 4, 1; bf16 ties at 1.0 go to the lower index 0
    assert list(O.topk(s, 2)) == [1, 4]
    assert list(O.topk(b, 2)) == [0, 4]
    assert list(O.topk(b, 3)) == [0, 1, 4]


def test_bf16_selection_and_recall():
    from csa2_synth import f32_to_bf16_bits
    rng = np.random.default_rng(1)
    n = 3000
    k = f32_to_bf16_bits(rng.standard_normal((n, 128)).astype(np.float32))
    q = f32_to_bf16_bits(rng.standard_normal((32, 128)).astype(np.float32))
    w = rng.standard_normal(32).astype(np.float32)
    idx, b, sc = O.index_topk_bf16(k, q, w, 512)
    full, _ = O.index_topk(k, q, w, 512)
    # brute force on the bf16 values: sort by (value desc, index asc)
    order = sorted(range(n), key=lambda i: (-float(b[i]), i))[:512]
    assert list(idx) == sorted(order)
    # every entry the fp32 selection keeps and the bf16 one drops sits in the
    # bf16 value of the 512-th score or within one bf16 step of it
    kth = sorted(b, reverse=True)[511]
    lost = set(full.tolist()) - set(idx.tolist())
    assert all(abs(float(b[i]) - float(kth)) <= abs(float(kth)) * 2.0 ** -7 for i in lost)
    r = O.recall(idx, full)
    assert r == 1.0 - len(lost) / 512
    assert O.recall(full, full) == 1.0
