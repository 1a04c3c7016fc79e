"""csa2_index_topk: queries at arbitrary token positions of several
sequences in one call (decode queries mixed with prefill positions), each
seeing the entries causally visible at its position ("DeepSeek-V4.1-Flash"
report, section 2.3.2), against the oracle; bf16 and MXFP4 indexer keys,
ratios 1 and 2, positions that see no entry, fewer than k entries, a ragged
block tail, and every entry."""
import numpy as np
import pytest

import csa2_synth as S
import oracle as O
from tests._parity import bf16_dev, check_topk, f32_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("idx_layout,ratio", [(0, 2), (0, 1), (1, 2)])
def test_mixed_positions_match_the_oracle(idx_layout, ratio):
    import fp4_kv_cache_index_gb300 as C
    lens = [2000, 513, 4096]
    cache = C.Cache(C.config(ratio=ratio, idx_layout=idx_layout), [4099, 515, 4096])
    ks = []
    for s, n in enumerate(lens):
        k = S.normal_bf16(S.stream_key(210, S.S_IDXK, s), 0, n * 128).reshape(n, 128)
        e = S.normal_f32(S.stream_key(210, S.S_ENTRIES, s), 0, n * 512).reshape(n, 512)
        C.csa2_append_entries(cache, [s], [n], f32_dev(e), bf16_dev(k))
        ks.append(k)
    m = ratio
    # (sequence, position): decode (last token), mid-sequence, before the
    # first complete block, fewer than k visible, a position past the last
    # appended entry (sees every entry), the odd position of a block
    queries = [(0, lens[0] * m - 1), (0, 1000), (1, 0), (1, 9), (2, 600 * m + m - 1),
               (2, 10 ** 7), (1, lens[1] * m - 1), (0, 1023 * m + m - 2), (2, 4095 * m)]
    nq = len(queries)
    qi = S.normal_bf16(S.stream_key(211, S.S_QIDX, 0), 0, nq * 4096).reshape(nq, 32, 128)
    w = S.normal_f32(S.stream_key(211, S.S_W, 0), 0, nq * 32).reshape(nq, 32)
    idx = C.csa2_index_topk(cache, bf16_dev(qi), f32_dev(w), [s for s, _ in queries],
                            [p for _, p in queries]).cpu().numpy()
    log = []
    for i, (s, p) in enumerate(queries):
        nv = O.visible_entries(lens[s], m, p)
        ref = O.index_topk_mxfp4 if idx_layout else O.index_topk
        o_idx, o_sc = ref(ks[s], qi[i], w[i], 512, nv)
        check_topk(idx[i], o_idx, o_sc if nv else np.zeros(1), 512, log)
        assert np.all(idx[i][idx[i] >= 0] < nv)
    assert cache.device_error() == 0
    print("near-ties:", log)


def test_negative_position_is_refused():
    import torch
    import fp4_kv_cache_index_gb300 as C
    cache = C.Cache(C.config(), [64])
    q = torch.zeros(1, 32, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(1, 32, device="cuda")
    with pytest.raises(C.Csa2Error):
        C.csa2_index_topk(cache, q, w, [0], [-1])
