"""csa2_index_topk_decode_static: the selection for callers that cannot
allocate device memory (scratch lives in a fixed array inside the library).
Its output must equal csa2_index_topk_decode's on the same inputs, on two
calls in a row (the second reuses the array the first left behind), and a
request larger than the array must be refused with nothing launched.

This file is collected last so that a failure here comes after every other
test has run."""
import ctypes

import numpy as np
import pytest

import csa2_synth as S
from tests._parity import bf16_dev, f32_dev

pytestmark = pytest.mark.gpu

CAPACITY = 3  # CSA2_ERR_CAPACITY


def _cache(C, lens, cap, seed):
    cache = C.Cache(C.config(), [cap] * len(lens))
    for s, n in enumerate(lens):
        k = S.normal_bf16(S.stream_key(seed, S.S_IDXK, s), 0, n * 128).reshape(n, 128)
        e = S.normal_f32(S.stream_key(seed, S.S_ENTRIES, s), 0, n * 512).reshape(n, 512)
        C.csa2_append_entries(cache, [s], [n], f32_dev(e), bf16_dev(k))
    return cache


def _static_call(C, cache, q_idx, w, seq_ids, idx_out, score_out):
    import torch
    ids = (ctypes.c_int32 * len(seq_ids))(*seq_ids) if seq_ids is not None else None
    return C.lib.csa2_index_topk_decode_static(
        cache.handle, q_idx.shape[0], ctypes.c_void_p(q_idx.data_ptr()),
        ctypes.c_void_p(w.data_ptr()), ids, ctypes.c_void_p(idx_out.data_ptr()),
        ctypes.c_void_p(score_out.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_static_scratch_matches_the_workspace_entry_point():
    import torch
    import fp4_kv_cache_index_gb300 as C
    lens = [20000, 513, 7000, 0, 16384]
    cache = _cache(C, lens, 20480, 61)
    for call, (seed, seq_ids) in enumerate([(62, None), (63, [4, 0, 0, 2, 1, 3])]):
        nq = len(seq_ids) if seq_ids is not None else len(lens)
        qi = S.normal_bf16(S.stream_key(seed, S.S_QIDX, 0), 0, nq * 4096).reshape(nq, 32, 128)
        w = S.normal_f32(S.stream_key(seed, S.S_W, 0), 0, nq * 32).reshape(nq, 32)
        q_idx, wd = bf16_dev(qi), f32_dev(w)
        ref_sc = torch.zeros(nq, 512, device="cuda")
        ref = C.csa2_index_topk_decode(cache, q_idx, wd, seq_ids, topk_score=ref_sc)
        got = torch.full((nq, 512), -7, dtype=torch.int32, device="cuda")
        got_sc = torch.full((nq, 512), 7.0, device="cuda")
        assert _static_call(C, cache, q_idx, wd, seq_ids, got, got_sc) == 0
        torch.cuda.synchronize()
        # same kernels, same arithmetic: identical selection and scores
        assert torch.equal(got, ref), f"call {call}"
        assert torch.equal(got_sc, ref_sc), f"call {call}"
    assert cache.device_error() == 0


def test_static_scratch_refuses_oversized_requests():
    import torch
    import fp4_kv_cache_index_gb300 as C
    cap = 1 << 21                       # 8 MiB of scores per query
    cache = C.Cache(C.config(), [cap])
    nq = 7                              # 7 x (8 MiB + 8 KiB) > 48 MiB
    q_idx = torch.zeros(nq, 32, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(nq, 32, device="cuda")
    idx = torch.full((nq, 512), -7, dtype=torch.int32, device="cuda")
    sc = torch.zeros(nq, 512, device="cuda")
    assert _static_call(C, cache, q_idx, w, [0] * nq, idx, sc) == CAPACITY
    torch.cuda.synchronize()
    assert torch.all(idx == -7)         # nothing was launched
