"""Micro-batched decode on two streams with a capped indexer grid
(csa2_cache_set_index_sms) gives bit-identical selections and readouts to
the whole batch on one stream: the schedule changes which SMs run what,
never the arithmetic."""
import numpy as np
import pytest

import csa2_synth as S
from tests._parity import bf16_dev, f32_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def C():
    import fp4_kv_cache_index_gb300 as C
    return C


def _setup(C, lens, seed):
    import torch
    cache = C.Cache(C.config(ratio=1), lens)
    for s, n in enumerate(lens):
        e = S.normal_f32(S.stream_key(seed, S.S_ENTRIES, s), 0, n * 512).reshape(n, 512)
        k = S.normal_bf16(S.stream_key(seed, S.S_IDXK, s), 0, n * 128).reshape(n, 128)
        C.csa2_append_entries(cache, [s], [n], f32_dev(e), bf16_dev(k))
    return cache


def _path(C, cache, q_idx, w, qs, swas, seq, lens, split, torch):
    n = len(seq)
    ld = (max(lens) + 3) // 4 * 4
    scores = torch.empty(n, ld, device="cuda")
    hist = torch.empty(n, 2048, dtype=torch.int32, device="cuda")
    topk = torch.empty(n, 512, dtype=torch.int32, device="cuda")
    tws = torch.empty(max(16, C.csa2_topk_workspace_bytes(n, max(lens))), dtype=torch.uint8,
                      device="cuda")
    aws = torch.empty(16 if split else 0, dtype=torch.uint8, device="cuda")
    C.csa2_index_scores_decode(cache, q_idx, w, scores, seq_ids=seq, key_hist=hist)
    C.csa2_topk(scores, [lens[s] for s in seq], 512, idx_out=topk, key_hist=hist, workspace=tws)
    outs, lses = [], []
    for q, swa in zip(qs, swas):
        lse = torch.empty(n, 64, device="cuda")
        outs.append(C.csa2_sparse_attn_decode(cache, q, swa, topk, 512 ** -0.5, seq_ids=seq,
                                              lse=lse, workspace=aws))
        lses.append(lse)
    return scores, topk, outs, lses


def test_micro_batches_match_one_stream(C):
    import torch
    lens = [3000, 5000, 700, 4100, 2600, 5120, 1500, 4999]
    cache = _setup(C, lens, 171)
    B, L = len(lens), 2
    q_idx = bf16_dev(S.normal_bf16(S.stream_key(172, S.S_QIDX, 0), 0, B * 4096).reshape(B, 32, 128))
    w = f32_dev(S.normal_f32(S.stream_key(172, S.S_W, 0), 0, B * 32).reshape(B, 32))
    qs = [bf16_dev(S.normal_bf16(S.stream_key(173, S.S_Q, l), 0, B * 64 * 512).reshape(B, 64, 512))
          for l in range(L)]
    swas = [bf16_dev(S.normal_bf16(S.stream_key(173, S.S_SWA, l), 0, B * 128 * 512)
                     .reshape(B, 128, 512)) for l in range(L)]
    whole = _path(C, cache, q_idx, w, qs, swas, list(range(B)), lens, True, torch)
    cache.set_index_sms(24)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    main = torch.cuda.current_stream()
    parts = []
    for m, s in enumerate(streams):
        s.wait_stream(main)
        lo, hi = B * m // 2, B * (m + 1) // 2
        with torch.cuda.stream(s):
            parts.append(_path(C, cache, q_idx[lo:hi].clone(), w[lo:hi].clone(),
                               [x[lo:hi].clone() for x in qs], [x[lo:hi].clone() for x in swas],
                               list(range(lo, hi)), lens, False, torch))
    for s in streams:
        main.wait_stream(s)
    torch.cuda.synchronize()
    cache.set_index_sms(0)
    sc, tk, outs, lses = whole
    # scores: each row's valid part (the tail of a row is not written)
    psc = torch.cat([p[0] for p in parts])
    for i, n in enumerate(lens):
        assert torch.equal(psc[i, :n], sc[i, :n])
    assert torch.equal(torch.cat([p[1] for p in parts]), tk)
    for l in range(L):
        # the unsplit readout of a micro-batch and the split one of the whole
        # batch merge their partial states in different orders: equal within
        # one bf16 step, and bit-equal to the whole batch read out unsplit
        a = torch.cat([p[2][l] for p in parts]).float()
        assert torch.allclose(a, outs[l].float(), rtol=2 ** -6, atol=1e-3)
    unsplit = _path(C, cache, q_idx, w, qs, swas, list(range(B)), lens, False, torch)
    for l in range(L):
        assert torch.equal(torch.cat([p[2][l] for p in parts]), unsplit[2][l])
        assert torch.equal(torch.cat([p[3][l] for p in parts]), unsplit[3][l])
    assert cache.device_error() == 0


def test_index_sms_argument(C):
    cache = C.Cache(C.config(), [64])
    with pytest.raises(C.Csa2Error):
        cache.set_index_sms(-1)
    cache.set_index_sms(0)
    cache.set_index_sms(100000)      # more than the GPU has: all of them
