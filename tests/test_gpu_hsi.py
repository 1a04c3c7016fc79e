"""GPU Hierarchical Sparse Indexer and Reindex mode ("DeepSeek-V4.1-Flash"
report, section 2.3.2) against the oracle.

* Pool: on the same fp32 scores (the GPU indexer's, copied to the host) the
  kept blocks are integer work and must equal the oracle's exactly; on the
  oracle's own fp64->fp32 scores they may differ only at near-ties of the
  block score.
* Reindex: on the same pool the selected positions follow the index-score
  parity rule (equal sets except near-ties of the k-th score), all inside the
  pool, ascending, -1 padded."""
import numpy as np
import pytest

import csa2_synth as S
import oracle as O
from tests._parity import bf16_dev, check_topk, f32_dev

pytestmark = pytest.mark.gpu

BLOCK = 8


@pytest.fixture(scope="module")
def C():
    import fp4_kv_cache_index_gb300 as C
    return C


def _fill(C, lens, cap, seed):
    cache = C.Cache(C.config(), [cap] * len(lens))
    ks = []
    for s, n in enumerate(lens):
        k = S.normal_bf16(S.stream_key(seed, S.S_IDXK, s), 0, n * 128).reshape(n, 128)
        e = S.normal_f32(S.stream_key(seed, S.S_ENTRIES, s), 0, n * 512).reshape(n, 512)
        if n:
            C.csa2_append_entries(cache, [s], [n], f32_dev(e), bf16_dev(k))
        ks.append(k)
    return cache, ks


def _queries(seed, nq):
    qi = S.normal_bf16(S.stream_key(seed, S.S_QIDX, 0), 0, nq * 4096).reshape(nq, 32, 128)
    w = S.normal_f32(S.stream_key(seed, S.S_W, 0), 0, nq * 32).reshape(nq, 32)
    return qi, w


def _full_scores(C, cache, qi, w, seq_ids, ld):
    import torch
    sc = torch.full((len(seq_ids), ld), float("nan"), device="cuda")
    C.csa2_index_scores_decode(cache, bf16_dev(qi), f32_dev(w), sc, seq_ids)
    return sc


def _check_pool_near_ties(gpu_pool, oracle_pool, oracle_block_scores):
    """Kept block sets equal except blocks whose oracle block score is within
    the near-tie distance of the oracle's last kept block score."""
    check_topk(gpu_pool, oracle_pool, oracle_block_scores, len(oracle_pool))


def _block_scores(sc64, n):
    nb = (n + BLOCK - 1) // BLOCK
    pad = np.full(nb * BLOCK, -np.inf)
    pad[:n] = sc64[:n]
    return pad.reshape(nb, BLOCK).max(axis=1)


@pytest.mark.parametrize("max_blocks", [2048, 64])
def test_pool_equals_oracle_on_the_same_scores(C, max_blocks):
    import torch
    lens = [20000, 16389, 3001, 0, 8, 16384]
    cache, ks = _fill(C, lens, 20480, 71)
    seq_ids = list(range(len(lens)))
    qi, w = _queries(72, len(seq_ids))
    ld = 20480
    sc = _full_scores(C, cache, qi, w, seq_ids, ld)
    pool = C.csa2_hsi_pool(sc, lens, max_blocks=max_blocks).cpu().numpy()
    sc_h = sc.cpu().numpy()
    for i, n in enumerate(lens):
        ref = O.hsi_pool(sc_h[i], n, BLOCK, max_blocks)
        assert np.array_equal(pool[i], ref), f"row {i} (n={n})"
    assert cache.device_error() == 0


def test_pool_against_the_oracles_scores(C):
    lens = [40000, 5000]
    cache, ks = _fill(C, lens, 40960, 73)
    qi, w = _queries(74, 2)
    sc = _full_scores(C, cache, qi, w, [0, 1], 40960)
    pool = C.csa2_hsi_pool(sc, lens, max_blocks=2048).cpu().numpy()
    for i, n in enumerate(lens):
        _, o_sc = O.index_topk(ks[i], qi[i], w[i], 512)
        bs = _block_scores(o_sc, n)
        o_pool = O.hsi_pool(o_sc.astype(np.float32), n, BLOCK, 2048)
        _check_pool_near_ties(pool[i], o_pool, bs)


@pytest.mark.parametrize("max_blocks", [2048, 48])
def test_reindex_matches_oracle(C, max_blocks):
    """Reindex selection against the oracle; 48 blocks = one tile of 32 and a
    half tile of 16, whose second half must write nothing (scores of the
    next query's row)."""
    import torch
    lens = [30000, 16384, 2000, 0, 20001]
    cache, ks = _fill(C, lens, 30720, 75)
    seq_ids = [0, 1, 2, 3, 4, 0, 4]
    nq = len(seq_ids)
    qf, wf = _queries(76, nq)            # the Full layer's indexer query
    qr, wr = _queries(77, nq)            # the Reindex layer's own query
    sc = _full_scores(C, cache, qf, wf, seq_ids, 30720)
    nv = [lens[s] for s in seq_ids]
    pool_d = C.csa2_hsi_pool(sc, nv, max_blocks=max_blocks)
    tsc = torch.full((nq, 512), 7.0, device="cuda")
    idx = C.csa2_index_topk_reindex_decode(cache, bf16_dev(qr), f32_dev(wr), pool_d,
                                           seq_ids, topk_score=tsc).cpu().numpy()
    pool = pool_d.cpu().numpy()
    tsc = tsc.cpu().numpy()
    log = []
    for i, s in enumerate(seq_ids):
        n = lens[s]
        o_idx, o_sc, pos = O.reindex_topk(ks[s], qr[i], wr[i], pool[i], n, 512, BLOCK)
        full = np.full(max(n, 1), -np.inf)
        full[pos] = o_sc
        check_topk(idx[i], o_idx, full, 512, log)
        valid = idx[i] >= 0
        assert set(idx[i][valid].tolist()) <= set(pos.tolist())
        if valid.any():
            ref = full[idx[i][valid]]
            assert np.allclose(tsc[i][valid], ref, rtol=2e-5, atol=2e-5 * np.abs(o_sc).max())
        assert np.all(tsc[i][~valid] == 0)
    assert cache.device_error() == 0
    print("near-ties:", log)


def test_small_context_reindex_equals_full_selection(C):
    """Fewer blocks than the pool holds: the pool is every entry and the
    Reindex selection is the Full selection of the same query, bit for bit
    (same scores on the same tensor-core tiles, same radix select)."""
    import torch
    lens = [12000, 700, 16384]
    cache, ks = _fill(C, lens, 16384, 78)
    qi, w = _queries(79, 3)
    sc = _full_scores(C, cache, qi, w, [0, 1, 2], 16384)
    pool_d = C.csa2_hsi_pool(sc, lens, max_blocks=2048)
    pool = pool_d.cpu().numpy()
    for i, n in enumerate(lens):
        nb = (n + BLOCK - 1) // BLOCK
        assert np.array_equal(pool[i][:nb], np.arange(nb))
        assert np.all(pool[i][nb:] == -1)
    s_full = torch.zeros(3, 512, device="cuda")
    s_re = torch.zeros(3, 512, device="cuda")
    full = C.csa2_index_topk_decode(cache, bf16_dev(qi), f32_dev(w), topk_score=s_full)
    re = C.csa2_index_topk_reindex_decode(cache, bf16_dev(qi), f32_dev(w), pool_d,
                                          topk_score=s_re)
    assert torch.equal(full, re)
    assert torch.equal(s_full, s_re)


def test_pool_smaller_than_k(C):
    """A pool of 16 blocks (128 positions) holds fewer than k = 512 entries:
    every pool position is selected, -1 padded."""
    lens = [5000]
    cache, ks = _fill(C, lens, 5120, 80)
    qf, wf = _queries(81, 1)
    qr, wr = _queries(82, 1)
    sc = _full_scores(C, cache, qf, wf, [0], 5120)
    pool_d = C.csa2_hsi_pool(sc, lens, max_blocks=16)
    idx = C.csa2_index_topk_reindex_decode(cache, bf16_dev(qr), f32_dev(wr), pool_d)
    pool = pool_d.cpu().numpy()[0]
    pos = O.pool_positions(pool, 5000)
    got = idx.cpu().numpy()[0]
    assert np.array_equal(got[:len(pos)], pos)
    assert np.all(got[len(pos):] == -1)


def test_reindex_unsupported_sizes_are_refused(C):
    import torch
    cache, _ = _fill(C, [100], 128, 83)
    q = torch.zeros(1, 32, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(1, 32, device="cuda")
    bad = torch.zeros(1, 24, dtype=torch.int32, device="cuda")   # not a multiple of 16
    with pytest.raises(C.Csa2Error):
        C.csa2_index_topk_reindex_decode(cache, q, w, bad)
    sc = torch.zeros(1, 128, device="cuda")
    with pytest.raises(C.Csa2Error):
        C.csa2_hsi_pool(sc, [100], max_blocks=24)
