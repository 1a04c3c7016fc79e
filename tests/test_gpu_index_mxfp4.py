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


def test_pool_mode_needs_bf16_keys(C):
    import torch
    cache, _ = _fill(C, [100], [100], 118)
    q = torch.zeros(1, 32, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(1, 32, device="cuda")
    pool = torch.zeros(1, 16, dtype=torch.int32, device="cuda")
    with pytest.raises(C.Csa2Error):
        C.csa2_index_topk_reindex_decode(cache, q, w, pool)


def test_out_of_range_scale_is_reported(C):
    """Keys around 2^20 need a block scale of 2^18, outside the E5M2 fast
    path's 2^-13 .. 2^13: the indexer clamps it and reports CSA2_ERR_DEVICE."""
    import torch
    n = 300
    cache = C.Cache(C.config(idx_layout=1), [n])
    k = S.normal_f32(S.stream_key(119, S.S_IDXK, 0), 0, n * 128).reshape(n, 128) * 2.0 ** 20
    e = S.normal_f32(S.stream_key(119, S.S_ENTRIES, 0), 0, n * 512).reshape(n, 512)
    C.csa2_append_entries(cache, [0], [n], f32_dev(e), bf16_dev(S.f32_to_bf16_bits(k)))
    assert cache.device_error() == 0
    qi, w = _queries(120, 1)
    C.csa2_index_topk_decode(cache, bf16_dev(qi), f32_dev(w))
    assert cache.device_error() == 7        # CSA2_ERR_DEVICE
