"""GPU indexer over MXFP4 indexer keys and queries ("DeepSeek-V4.1-Flash"
report, section 2.4.4) against the oracle: the appended key codes and
scales bit-exact, the scores close to the fp64 score of the rounded inputs,
top-k sets equal except logged near-ties; ragged sequences whose offsets
are not multiples of 4 (the scale windows) and a tile that ends at the end
of the cache; decode, prefill and bf16-rounded scores."""
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


def _fill(C, lens, caps, seed, ratio=1):
    cache = C.Cache(C.config(ratio=ratio, idx_layout=1), caps)
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


# capacities 1001, 3, 2047, 514: sequence offsets 0, 1001, 1004, 3051 (not
# multiples of 4); the last sequence fills its capacity, so its last tile
# ends at the end of the cache
LENS = [1001, 2, 2047, 514]
CAPS = [1001, 3, 2047, 514]


def test_appended_keys_are_the_oracles_mxfp4(C):
    cache, ks = _fill(C, LENS, CAPS, 111)
    v = cache.views()
    assert v["idx_k"] is None
    codes = v["idx_codes"].cpu().numpy()
    scales = v["idx_scales"].cpu().numpy()
    for s, n in enumerate(LENS):
        o = v["entry_offset"][s]
        oc, os_ = O.quantise(S.bf16_bits_to_f32(ks[s]), O.LAYOUT_L32_UE8M0)
        assert np.array_equal(codes[o:o + n], oc)
        assert np.array_equal(scales[o:o + n], os_)
    assert cache.device_error() == 0


def test_decode_scores_and_selection(C):
    import torch
    cache, ks = _fill(C, LENS, CAPS, 112)
    seq_ids = [0, 1, 2, 3, 3, 0]
    nq = len(seq_ids)
    qi, w = _queries(113, nq)
    ld = 2048
    sc = torch.full((nq, ld), float("nan"), device="cuda")
    C.csa2_index_scores_decode(cache, bf16_dev(qi), f32_dev(w), sc, seq_ids)
    sc = sc.cpu().numpy()
    tsc = torch.zeros(nq, 512, device="cuda")
    idx = C.csa2_index_topk_decode(cache, bf16_dev(qi), f32_dev(w), seq_ids,
                                   topk_score=tsc).cpu().numpy()
    tsc = tsc.cpu().numpy()
    log = []
    for i, s in enumerate(seq_ids):
        n = LENS[s]
        o_idx, o_sc = O.index_topk_mxfp4(ks[s], qi[i], w[i], 512)
        assert np.allclose(sc[i, :n], o_sc, rtol=2e-5, atol=2e-5 * np.abs(o_sc).max())
        assert np.all(np.isnan(sc[i, n:]))
        check_topk(idx[i], o_idx, o_sc, 512, log)
        ok = idx[i] >= 0
        assert np.array_equal(tsc[i][ok], sc[i][idx[i][ok]])
    assert cache.device_error() == 0
    print("near-ties:", log)


def test_bf16_scores_on_mxfp4_keys(C):
    import torch
    cache, ks = _fill(C, LENS, CAPS, 114)
    qi, w = _queries(115, 4)
    s32 = torch.zeros(4, 2048, device="cuda")
    s16 = torch.zeros(4, 2048, dtype=torch.bfloat16, device="cuda")
    C.csa2_index_scores_decode(cache, bf16_dev(qi), f32_dev(w), s32)
    C.csa2_index_scores_decode_bf16(cache, bf16_dev(qi), f32_dev(w), s16)
    a = s32.cpu().numpy()
    b = S.bf16_bits_to_f32(s16.view(torch.int16).cpu().numpy().view(np.uint16))
    for i, n in enumerate(LENS):
        assert np.array_equal(b[i, :n], O.bf16_round(a[i, :n]))


@pytest.mark.parametrize("pos0,ratio", [(1900, 2), (0, 1), (2999, 1)])
def test_prefill_causal(C, pos0, ratio):
    n_ent = 1000 if ratio == 2 else 3000
    cache, ks = _fill(C, [n_ent], [n_ent + 3], 116, ratio=ratio)
    nq = 37
    qi, w = _queries(117, nq)
    idx = C.csa2_index_topk_prefill(cache, 0, pos0, bf16_dev(qi), f32_dev(w)).cpu().numpy()
    for i in range(nq):
        nv = O.visible_entries(n_ent, ratio, pos0 + i)
        o_idx, o_sc = O.index_topk_mxfp4(ks[0], qi[i], w[i], 512, nv)
        check_topk(idx[i], o_idx, o_sc, 512)
    assert cache.device_error() == 0


def test_prefill_histograms_need_bf16_keys(C):
    """The prefill score-key histograms come from the bf16 indexer only: with
    MXFP4 keys the request is refused (the selection above builds its own)."""
    import torch
    cache, _ = _fill(C, [600], [600], 118)
    qi, w = _queries(119, 4)
    sc = torch.empty(4, 600, device="cuda")
    kh = torch.zeros(4, 2048, dtype=torch.int32, device="cuda")
    with pytest.raises(C.Csa2Error, match="UNSUPPORTED"):
        C.csa2_index_scores_prefill(cache, 0, 700, bf16_dev(qi), f32_dev(w), sc, key_hist=kh)
    C.csa2_index_scores_prefill(cache, 0, 700, bf16_dev(qi), f32_dev(w), sc)
    assert cache.device_error() == 0


def _reindex_case(C, lens, cap, seq_ids, max_blocks, seed):
    """Full-layer scores over MXFP4 keys -> candidate pool -> Reindex selection
    with another query, against the oracle on the MXFP4-rounded keys and
    queries."""
    import torch
    cache, ks = _fill(C, lens, [cap] * len(lens), seed)
    nq = len(seq_ids)
    qf, wf = _queries(seed + 1, nq)            # the Full layer's indexer query
    qr, wr = _queries(seed + 2, nq)            # the Reindex layer's own query
    sc = torch.full((nq, (cap + 3) // 4 * 4), float("nan"), device="cuda")
    C.csa2_index_scores_decode(cache, bf16_dev(qf), f32_dev(wf), sc, seq_ids)
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
        kq = O.mxfp4_round_bf16(ks[s][:n])
        qq = O.mxfp4_round_bf16(qr[i])
        o_idx, o_sc, pos = O.reindex_topk(kq, qq, wr[i], pool[i], n, 512)
        full = np.full(max(n, 1), -np.inf)
        full[pos] = o_sc
        check_topk(idx[i], o_idx, full, 512, log)
        valid = idx[i] >= 0
        assert set(idx[i][valid].tolist()) <= set(pos.tolist())
        if valid.any():
            assert np.allclose(tsc[i][valid], full[idx[i][valid]], rtol=2e-5,
                               atol=2e-5 * np.abs(o_sc).max())
        assert np.all(tsc[i][~valid] == 0)
    assert cache.device_error() == 0
    return log


def test_reindex_on_mxfp4_keys(C):
    """Reindex mode ("DeepSeek-V4.1-Flash" report, section 2.3.2) over the
    report's FP4 indexer keys (section 2.4.4): pools of 2048 blocks of 8
    over ragged sequences whose offsets are not multiples of 4."""
    log = _reindex_case(C, [30000, 16384, 2000, 0, 20001], 30721, [0, 1, 2, 3, 4, 0, 4],
                        2048, 130)
    print("near-ties:", log)


@pytest.mark.parametrize("max_blocks", [48, 80])
def test_reindex_on_mxfp4_keys_partial_tile(C, max_blocks):
    """Pools of 48 and 80 blocks: the last 512-slot tile of the MXFP4 indexer
    holds 48 or 16 blocks (slots past the pool are neither scored nor
    stored)."""
    _reindex_case(C, [3000, 777], 3001, [0, 1, 1], max_blocks, 140)


def test_small_context_reindex_equals_full_selection_mxfp4(C):
    """Fewer blocks than the pool holds: the Reindex selection equals the
    Full selection of the same query on the same MXFP4 keys, bit for bit."""
    import torch
    lens = [12000, 700, 16384]
    cache, ks = _fill(C, lens, [16384] * 3, 150)
    qi, w = _queries(151, 3)
    sc = torch.full((3, 16384), float("nan"), device="cuda")
    C.csa2_index_scores_decode(cache, bf16_dev(qi), f32_dev(w), sc)
    pool_d = C.csa2_hsi_pool(sc, lens, max_blocks=2048)
    s_full = torch.zeros(3, 512, device="cuda")
    s_re = torch.zeros(3, 512, device="cuda")
    full = C.csa2_index_topk_decode(cache, bf16_dev(qi), f32_dev(w), topk_score=s_full)
    re = C.csa2_index_topk_reindex_decode(cache, bf16_dev(qi), f32_dev(w), pool_d,
                                          topk_score=s_re)
    assert torch.equal(full, re)
    assert torch.equal(s_full, s_re)


@pytest.mark.parametrize("mag", [2.0 ** 20, 2.0 ** -20])
def test_extreme_block_scales(C, mag):
    """Keys around 2^20 (block scale 2^18) or 2^-20 (2^-22): the block-scaled
    MMAs take any UE8M0 scale, so the scores still match the oracle's fp64
    score of the rounded values and nothing is flagged."""
    import torch
    n = 3000
    cache = C.Cache(C.config(idx_layout=1), [n])
    k = S.normal_f32(S.stream_key(119, S.S_IDXK, 0), 0, n * 128).reshape(n, 128) * mag
    kb = S.f32_to_bf16_bits(k)
    e = S.normal_f32(S.stream_key(119, S.S_ENTRIES, 0), 0, n * 512).reshape(n, 512)
    C.csa2_append_entries(cache, [0], [n], f32_dev(e), bf16_dev(kb))
    qi, w = _queries(120, 2)
    sc = torch.full((2, n), float("nan"), device="cuda")
    C.csa2_index_scores_decode(cache, bf16_dev(qi), f32_dev(w), sc, [0, 0])
    sc = sc.cpu().numpy()
    idx = C.csa2_index_topk_decode(cache, bf16_dev(qi), f32_dev(w), [0, 0]).cpu().numpy()
    for i in range(2):
        o_idx, o_sc = O.index_topk_mxfp4(kb, qi[i], w[i], 512)
        assert np.allclose(sc[i], o_sc, rtol=2e-5, atol=2e-5 * np.abs(o_sc).max())
        check_topk(idx[i], o_idx, o_sc, 512)
    assert cache.device_error() == 0
