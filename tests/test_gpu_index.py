"""GPU indexer + top-k (tcgen05 score kernel, radix select) against the
oracle: fp64 scores rounded to fp32, top-k sets equal except logged
near-ties within 1e-5 of the k-th score; returned scores close to fp64."""
import numpy as np
import pytest

import csa2_synth as S
import oracle as O
from tests._parity import bf16_dev, check_topk, f32_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def C():
    import fp4_kv_cache_index_gb300 as C
    return C


def _fill(C, lens, cap, seed, ratio=1):
    cache = C.Cache(C.config(ratio=ratio), [cap] * len(lens))
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


def test_decode_ragged_and_shared_sequences(C):
    import torch
    lens = [0, 100, 511, 513, 3000, 1280]
    cache, ks = _fill(C, lens, 3072, 21)
    seq_ids = [0, 1, 2, 3, 4, 5, 4, 4]
    qi, w = _queries(22, len(seq_ids))
    sc = torch.zeros(len(seq_ids), 512, dtype=torch.float32, device="cuda")
    idx = C.csa2_index_topk_decode(cache, bf16_dev(qi), f32_dev(w), seq_ids, topk_score=sc)
    idx = idx.cpu().numpy()
    sc = sc.cpu().numpy()
    log = []
    for i, s in enumerate(seq_ids):
        o_idx, o_sc = O.index_topk(ks[s], qi[i], w[i], 512)
        check_topk(idx[i], o_idx, o_sc, 512, log)
        valid = idx[i] >= 0
        if valid.any():
            ref = o_sc[idx[i][valid]]
            assert np.allclose(sc[i][valid], ref, rtol=2e-5, atol=2e-5 * np.abs(o_sc).max())
        assert np.all(sc[i][~valid] == 0)
    assert cache.device_error() == 0
    print("near-ties:", log)


def test_zero_query_selects_first_k(C):
    cache, ks = _fill(C, [2000], 2048, 23)
    qi = np.zeros((1, 32, 128), np.uint16)
    w = np.ones((1, 32), np.float32)
    idx = C.csa2_index_topk_decode(cache, bf16_dev(qi), f32_dev(w)).cpu().numpy()[0]
    assert np.array_equal(idx, np.arange(512))


def test_single_head_is_relu_dot(C):
    cache, ks = _fill(C, [1500], 1536, 24)
    qi, _ = _queries(25, 1)
    w = np.zeros((1, 32), np.float32)
    w[0, 5] = 1.0
    idx = C.csa2_index_topk_decode(cache, bf16_dev(qi), f32_dev(w)).cpu().numpy()[0]
    o_idx, o_sc = O.index_topk(ks[0], qi[0], w[0], 512)
    # many entries have ReLU(.) = 0: the k-th score may be a tie at 0
    check_topk(idx, o_idx, o_sc, 512)


@pytest.mark.parametrize("pos0,ratio", [(1900, 2), (700, 2), (0, 1), (2999, 1)])
def test_prefill_causal(C, pos0, ratio):
    n_ent = 1000 if ratio == 2 else 3000
    cache, ks = _fill(C, [n_ent], 3072, 26, ratio=ratio)
    nq = 37
    qi, w = _queries(27, nq)
    idx = C.csa2_index_topk_prefill(cache, 0, pos0, bf16_dev(qi), f32_dev(w)).cpu().numpy()
    for i in range(nq):
        nv = O.visible_entries(n_ent, ratio, pos0 + i)
        o_idx, o_sc = O.index_topk(ks[0], qi[i], w[i], 512, nv)
        check_topk(idx[i], o_idx, o_sc, 512)


def test_prefill_scores_and_key_histogram(C):
    """csa2_index_scores_prefill with score-key histograms (eight queries per
    tile, each with its own histogram): every query's histogram exactly that
    of its visible scores, across a chunk whose queries straddle groups of
    eight and see different numbers of entries, and the top-k from the
    histograms identical to the top-k without them."""
    import torch
    n_ent, ratio, pos0, nq = 3000, 2, 5000, 45
    cache, ks = _fill(C, [n_ent], 3072, 28, ratio=ratio)
    qi, w = _queries(29, nq)
    ld = 3072
    sc = torch.full((nq, ld), float("nan"), device="cuda")
    kh = torch.full((nq, 2048), 7, dtype=torch.int32, device="cuda")   # zeroed by the call
    C.csa2_index_scores_prefill(cache, 0, pos0, bf16_dev(qi), f32_dev(w), sc, key_hist=kh)
    sc_h, kh_h = sc.cpu().numpy(), kh.cpu().numpy()
    nv = [O.visible_entries(n_ent, ratio, pos0 + i) for i in range(nq)]
    assert len(set(nv)) > 1
    for i in range(nq):
        assert np.all(np.isnan(sc_h[i, nv[i]:]))
        assert np.array_equal(kh_h[i], _key_hist(sc_h[i, :nv[i]])), i
    a = C.csa2_topk(sc, nv, 512, key_hist=kh).cpu().numpy()
    b = C.csa2_topk(sc, nv, 512).cpu().numpy()
    assert np.array_equal(a, b)


def _key_hist(scores):
    u = np.ascontiguousarray(scores, np.float32).view(np.uint32).copy()
    u[(u << np.uint32(1)) == 0] = 0
    key = np.where(u & np.uint32(0x80000000), ~u, u | np.uint32(0x80000000))
    return np.bincount((key >> np.uint32(21)).astype(np.int64), minlength=2048)


def test_scores_and_key_histogram(C):
    """csa2_index_scores_decode: every score close to the fp64 oracle, the
    score-key histogram exactly that of the returned scores, and top-k from
    the histogram identical to top-k without it."""
    import torch
    lens = [5000, 0, 700, 3001]
    cache, ks = _fill(C, lens, 5120, 41)
    qi, w = _queries(42, len(lens))
    ld = 5120
    sc = torch.full((len(lens), ld), float("nan"), device="cuda")
    kh = torch.zeros(len(lens), 2048, dtype=torch.int32, device="cuda")
    C.csa2_index_scores_decode(cache, bf16_dev(qi), f32_dev(w), sc, key_hist=kh)
    sc_h, kh_h = sc.cpu().numpy(), kh.cpu().numpy()
    for i, n in enumerate(lens):
        assert np.all(np.isnan(sc_h[i, n:]))          # past the length: untouched
        if n:
            o = O.index_scores(ks[i], qi[i], w[i])
            assert np.allclose(sc_h[i, :n], o, rtol=2e-5, atol=2e-5 * np.abs(o).max())
        assert np.array_equal(kh_h[i], _key_hist(sc_h[i, :n]))
    a = C.csa2_topk(sc, lens, 512, key_hist=kh).cpu().numpy()
    b = C.csa2_topk(sc, lens, 512).cpu().numpy()
    assert np.array_equal(a, b)
    for i, n in enumerate(lens):
        assert np.array_equal(a[i], O.topk(sc_h[i, :n], 512))
