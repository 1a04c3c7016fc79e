"""Pins of the oracle's Hierarchical Sparse Indexer and Reindex mode
("DeepSeek-V4.1-Flash" report, section 2.3.2: block score = maximum index
score of its positions, the highest blocks form the candidate pool -- 2,048
blocks of 8 positions give 16,384 candidates -- and Reindex layers select
their own top-k inside the pool)."""
import numpy as np
import pytest

import oracle as O
from csa2_synth import f32_to_bf16_bits
from tests._golden import numbers

G = numbers()


def test_pool_size_from_the_pages():
    s = np.random.default_rng(0).standard_normal(1 << 16).astype(np.float32)
    pool = O.hsi_pool(s, len(s), G["hsi_block_positions"], G["hsi_blocks"])
    assert (pool >= 0).sum() == G["hsi_blocks"]
    assert len(O.pool_positions(pool, len(s), G["hsi_block_positions"])) == G["hsi_pool"]


def test_block_scores_brute_force():
    rng = np.random.default_rng(1)
    n = 203                                    # ragged last block
    s = rng.integers(-5, 5, n).astype(np.float32)
    pool = O.hsi_pool(s, n, 8, 7)
    bmax = [s[b * 8:b * 8 + 8].max() for b in range((n + 7) // 8)]
    order = sorted(range(len(bmax)), key=lambda b: (-bmax[b], b))[:7]
    assert list(pool) == sorted(order)


def test_small_context_pool_is_everything_and_reindex_equals_full():
    """With no more blocks than the pool holds, the pool is every visible
    position, and a Reindex layer selects exactly what a Full layer with the
    same indexer query would."""
    rng = np.random.default_rng(2)
    n = 3001
    k = f32_to_bf16_bits(rng.standard_normal((n, 128)).astype(np.float32))
    q = f32_to_bf16_bits(rng.standard_normal((32, 128)).astype(np.float32))
    w = rng.standard_normal(32).astype(np.float32)
    full_idx, full_sc = O.index_topk(k, q, w, 512)
    pool = O.hsi_pool(full_sc.astype(np.float32), n, 8, 2048)
    assert np.array_equal(O.pool_positions(pool, n), np.arange(n))
    q2 = f32_to_bf16_bits(rng.standard_normal((32, 128)).astype(np.float32))
    re_idx, _, _ = O.reindex_topk(k, q2, w, pool, n)
    assert np.array_equal(re_idx, O.index_topk(k, q2, w, 512)[0])


def test_pool_contains_the_full_layers_selection():
    """Every block holding one of the Full layer's top-k entries has a block
    score at least the k-th score, so it is in the pool when the pool keeps
    at least k blocks."""
    rng = np.random.default_rng(3)
    n = 40000
    s = rng.standard_normal(n).astype(np.float32)
    top = O.topk(s, 512)
    pool = O.hsi_pool(s, n, 8, 2048)
    assert set(top.tolist()) <= set(O.pool_positions(pool, n).tolist())


def test_reindex_is_restricted_to_the_pool():
    rng = np.random.default_rng(4)
    n = 50000
    k = f32_to_bf16_bits(rng.standard_normal((n, 128)).astype(np.float32))
    q = f32_to_bf16_bits(rng.standard_normal((32, 128)).astype(np.float32))
    w = rng.standard_normal(32).astype(np.float32)
    s = rng.standard_normal(n).astype(np.float32)     # some other layer's scores
    pool = O.hsi_pool(s, n, 8, 256)                   # 2048 positions
    idx, sc, pos = O.reindex_topk(k, q, w, pool, n)
    assert set(idx.tolist()) <= set(pos.tolist())
    # brute force over the pool positions
    scf = sc.astype(np.float32)
    order = sorted(range(len(pos)), key=lambda i: (-float(scf[i]), int(pos[i])))[:512]
    assert list(idx) == sorted(int(pos[i]) for i in order)
