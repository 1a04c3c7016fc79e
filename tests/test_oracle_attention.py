"""Pins of the oracle's sparse shared-KV attention with the sliding window
(blog reading of the DeepSeek-V4 report, sections 4.1 and 4.3; neshdevtech
article section 3.3.1 "Readout concatenates the SWA and the selected Main KV
into a single joint sparse attention", section 3.3.2.1 convex combination)."""
import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import oracle as O
from csa2_synth import bf16_bits_to_f32, f32_to_bf16_bits

L = O.LAYOUT_L32_UE8M0


def _case(rng, heads=8, dim=64, n=40, n_swa=6):
    q = f32_to_bf16_bits(rng.standard_normal((heads, dim)).astype(np.float32))
    codes, scales = O.quantise(rng.standard_normal((n, dim)).astype(np.float32), L)
    swa = f32_to_bf16_bits(rng.standard_normal((n_swa, dim)).astype(np.float32))
    return q, codes, scales, swa


def test_all_selected_equals_dense_softmax_attention():
    rng = np.random.default_rng(0)
    q, codes, scales, swa = _case(rng)
    scale = 1 / np.sqrt(64)
    idx = np.arange(40, dtype=np.int32)
    _, out, lse = O.sparse_attention(q, codes, scales, L, idx, swa, scale)
    kv = np.concatenate([O.dequantise(codes, scales, L).astype(np.float64),
                         bf16_bits_to_f32(swa).astype(np.float64)])
    logits = np.float64(np.float32(scale)) * (bf16_bits_to_f32(q).astype(np.float64) @ kv.T)
    assert np.allclose(out, softmax(logits, axis=1) @ kv, rtol=1e-12, atol=1e-13)
    assert np.allclose(lse, logsumexp(logits, axis=1), rtol=1e-12)


def test_lse_merge_of_the_two_branches_is_the_joint_softmax():
    rng = np.random.default_rng(1)
    q, codes, scales, swa = _case(rng)
    idx = rng.choice(40, 16, replace=False).astype(np.int32)
    _, o_all, l_all = O.sparse_attention(q, codes, scales, L, idx, swa, 0.125)
    _, o_s, l_s = O.sparse_attention(q, codes, scales, L, idx, None, 0.125)
    _, o_w, l_w = O.sparse_attention(q, codes, scales, L, np.zeros(0, np.int32), swa, 0.125)
    lse = np.logaddexp(l_s, l_w)
    merged = (np.exp(l_s - lse)[:, None] * o_s + np.exp(l_w - lse)[:, None] * o_w)
    assert np.allclose(l_all, lse, rtol=1e-12)
    assert np.allclose(o_all, merged, rtol=1e-10, atol=1e-12)


def test_output_is_in_the_convex_hull():
    rng = np.random.default_rng(2)
    q, codes, scales, swa = _case(rng, n=100)
    idx = np.arange(0, 100, 3, dtype=np.int32)
    _, out, _ = O.sparse_attention(q, codes, scales, L, idx, swa, 0.3)
    kv = np.concatenate([O.dequantise(codes[idx], scales[idx], L), bf16_bits_to_f32(swa)])
    assert np.all(out <= kv.max(axis=0) + 1e-12) and np.all(out >= kv.min(axis=0) - 1e-12)


def test_zero_query_gives_the_uniform_mean():
    rng = np.random.default_rng(3)
    _, codes, scales, swa = _case(rng)
    q = np.zeros((8, 64), np.uint16)
    idx = np.array([3, 5, 7, -1, -1], np.int32)
    _, out, lse = O.sparse_attention(q, codes, scales, L, idx, swa, 1.0)
    kv = np.concatenate([O.dequantise(codes[[3, 5, 7]], scales[[3, 5, 7]], L),
                         bf16_bits_to_f32(swa)]).astype(np.float64)
    assert np.allclose(out, np.tile(kv.mean(axis=0), (8, 1)), rtol=1e-13, atol=1e-15)
    assert np.allclose(lse, np.log(9.0))


def test_padding_and_order_do_not_matter():
    rng = np.random.default_rng(4)
    q, codes, scales, swa = _case(rng)
    a = O.sparse_attention(q, codes, scales, L, np.array([1, 9, 30], np.int32), swa, 0.2)
    b = O.sparse_attention(q, codes, scales, L, np.array([30, -1, 1, -1, 9], np.int32), swa, 0.2)
    assert np.allclose(a[1], b[1], rtol=1e-13) and np.array_equal(a[0], b[0])


def test_single_candidate_returns_it():
    rng = np.random.default_rng(5)
    q, codes, scales, _ = _case(rng)
    ob, od, lse = O.sparse_attention(q, codes, scales, L, np.array([11], np.int32), None, 0.5)
    kv = O.dequantise(codes[[11]], scales[[11]], L)[0].astype(np.float64)
    assert np.array_equal(od, np.tile(kv, (8, 1)))
    assert np.array_equal(bf16_bits_to_f32(ob), np.tile(kv.astype(np.float32), (8, 1)))  # -0 == +0
    assert np.allclose(lse, 0.5 * (bf16_bits_to_f32(q).astype(np.float64) @ kv))
