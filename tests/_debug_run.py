"""Parity cases run under the bounds-checked library (libcsa2_debug.so).
Executed as a script by tests/test_gpu_debug_build.py in a child process
with CSA2_DEBUG=1: decode selection and readout (both main-KV layouts,
bf16 and MXFP4 indexer keys), Reindex, prefill, each against the oracle
with the device error word clean; then a top-k row holding an index past
the sequence, which must be reported as CSA2_ERR_DEVICE."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import csa2_synth as S  # noqa: E402
import fp4_kv_cache_index_gb300 as C  # noqa: E402
import oracle as O  # noqa: E402
from tests._parity import bf16_dev, bf16_host, check_attn, check_topk, f32_dev  # noqa: E402


def fill(cfg, lens, cap, seed):
    cache = C.Cache(cfg, [cap] * len(lens))
    ks, es = [], []
    for s, n in enumerate(lens):
        k = S.normal_bf16(S.stream_key(seed, S.S_IDXK, s), 0, n * 128).reshape(n, 128)
        e = S.normal_f32(S.stream_key(seed, S.S_ENTRIES, s), 0, n * 512).reshape(n, 512)
        C.csa2_append_entries(cache, [s], [n], f32_dev(e), bf16_dev(k))
        ks.append(k)
        es.append(e)
    return cache, ks, es


def decode(layout, idx_layout, seed):
    lens = [3000, 700, 1501]
    cache, ks, es = fill(C.config(layout=layout, idx_layout=idx_layout), lens, 3001, seed)
    nq = len(lens)
    qi = S.normal_bf16(S.stream_key(seed + 1, S.S_QIDX, 0), 0, nq * 4096).reshape(nq, 32, 128)
    w = S.normal_f32(S.stream_key(seed + 1, S.S_W, 0), 0, nq * 32).reshape(nq, 32)
    q = S.normal_bf16(S.stream_key(seed + 1, S.S_Q, 0), 0, nq * 64 * 512).reshape(nq, 64, 512)
    swa = S.normal_bf16(S.stream_key(seed + 1, S.S_SWA, 0), 0, nq * 128 * 512).reshape(nq, 128, 512)
    idx = C.csa2_index_topk_decode(cache, bf16_dev(qi), f32_dev(w))
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    out = C.csa2_sparse_attn_decode(cache, bf16_dev(q), bf16_dev(swa), idx, 512 ** -0.5,
                                    workspace=ws)
    idx_h = idx.cpu().numpy()
    out_h = bf16_host(out)
    for i, n in enumerate(lens):
        ref = O.index_topk_mxfp4 if idx_layout else O.index_topk
        o_idx, o_sc = ref(ks[i], qi[i], w[i], 512)
        check_topk(idx_h[i], o_idx, o_sc, 512)
        codes, scales = O.quantise(es[i], layout)
        _, o_out, _ = O.sparse_attention(q[i], codes, scales, layout, idx_h[i], swa[i],
                                         np.float32(512 ** -0.5))
        check_attn(out_h[i], o_out)
    assert cache.device_error() == 0, "debug checks fired on a valid decode"
    # Reindex over the same cache
    sc = torch.full((nq, 3004), float("nan"), device="cuda")
    C.csa2_index_scores_decode(cache, bf16_dev(qi), f32_dev(w), sc)
    pool = C.csa2_hsi_pool(sc, lens, max_blocks=64)
    re = C.csa2_index_topk_reindex_decode(cache, bf16_dev(qi), f32_dev(w), pool).cpu().numpy()
    pool_h = pool.cpu().numpy()
    for i, n in enumerate(lens):
        kk = O.mxfp4_round_bf16(ks[i]) if idx_layout else ks[i]
        qq = O.mxfp4_round_bf16(qi[i]) if idx_layout else qi[i]
        o_idx, o_sc, pos = O.reindex_topk(kk, qq, w[i], pool_h[i], n, 512)
        full = np.full(n, -np.inf)
        full[pos] = o_sc
        check_topk(re[i], o_idx, full, 512)
    assert cache.device_error() == 0, "debug checks fired on a valid Reindex"


def prefill(seed):
    n_ent, pos0, nq = 1000, 1900, 40
    cache, ks, es = fill(C.config(ratio=2), [n_ent], n_ent + 5, seed)
    qi = S.normal_bf16(S.stream_key(seed + 1, S.S_QIDX, 0), 0, nq * 4096).reshape(nq, 32, 128)
    w = S.normal_f32(S.stream_key(seed + 1, S.S_W, 0), 0, nq * 32).reshape(nq, 32)
    idx = C.csa2_index_topk_prefill(cache, 0, pos0, bf16_dev(qi), f32_dev(w)).cpu().numpy()
    for i in range(nq):
        nv = O.visible_entries(n_ent, 2, pos0 + i)
        o_idx, o_sc = O.index_topk(ks[0], qi[i], w[i], 512, nv)
        check_topk(idx[i], o_idx, o_sc, 512)
    assert cache.device_error() == 0, "debug checks fired on a valid prefill"


def bad_index(seed):
    cache, _, _ = fill(C.config(), [600], 600, seed)
    q = torch.zeros(1, 64, 512, dtype=torch.bfloat16, device="cuda")
    swa = torch.zeros(1, 128, 512, dtype=torch.bfloat16, device="cuda")
    idx = torch.full((1, 512), -1, dtype=torch.int32, device="cuda")
    idx[0, 3] = 600                                  # one past the sequence
    C.csa2_sparse_attn_decode(cache, q, swa, idx, 512 ** -0.5)
    assert cache.device_error() == 7                 # CSA2_ERR_DEVICE


if __name__ == "__main__":
    assert C.LIB_PATH.endswith("libcsa2_debug.so"), C.LIB_PATH
    decode(0, 0, 170)
    decode(1, 1, 180)
    prefill(190)
    bad_index(200)
    print("debug build: all cases clean")
