"""GPU sparse attention (FP4 gather-dequant + tcgen05 QK^T / PV + window +
joint softmax) against the oracle's fp64 attention: max-abs 1e-2 and
mean-abs 1e-3 on the bf16 outputs, lse within 1e-3."""
import numpy as np
import pytest

import csa2_synth as S
import oracle as O
from tests._parity import bf16_dev, bf16_host, check_attn, f32_dev, check_lse

pytestmark = pytest.mark.gpu
SCALE = np.float32(512 ** -0.5)


@pytest.fixture(scope="module")
def C():
    import fp4_kv_cache_index_gb300 as C
    return C


def _cache(C, lens, cap, seed, layout=0, ratio=1, outlier=None):
    cache = C.Cache(C.config(layout=layout, ratio=ratio), [cap] * len(lens))
    ents = []
    for s, n in enumerate(lens):
        e = S.normal_f32(S.stream_key(seed, S.S_ENTRIES, s), 0, n * 512).reshape(n, 512)
        if outlier is not None:
            e[:, outlier] *= 8
        k = S.normal_bf16(S.stream_key(seed, S.S_IDXK, s), 0, n * 128).reshape(n, 128)
        if n:
            C.csa2_append_entries(cache, [s], [n], f32_dev(e), bf16_dev(k))
        ents.append(e)
    return cache, ents


def _sel(rng, n, k=512, fill=None):
    m = min(n, k) if fill is None else fill
    idx = np.sort(rng.choice(n, m, replace=False)) if m else np.zeros(0, np.int64)
    out = np.full(k, -1, np.int32)
    out[:m] = idx
    return out


@pytest.mark.parametrize("layout", [0, 1])
def test_decode_matches_oracle(C, layout):
    import torch
    rng = np.random.default_rng(layout)
    lens = [700, 300, 1000, 5000]
    outl = np.array([3, 77, 200, 301, 511])
    cache, ents = _cache(C, lens, 5120, 31, layout, outlier=outl)
    nq = len(lens)
    q = S.normal_bf16(S.stream_key(32, S.S_Q, 0), 0, nq * 64 * 512).reshape(nq, 64, 512)
    swa = S.normal_f32(S.stream_key(32, S.S_SWA, 0), 0, nq * 128 * 512).reshape(nq, 128, 512)
    swa[..., outl] *= 8
    swa = S.f32_to_bf16_bits(swa)
    swa_len = np.array([128, 50, 0, 1], np.int32)
    idx = np.stack([_sel(rng, n) for n in lens])
    idx[3, 100:] = -1                      # a query with 100 selected entries only
    lse = torch.zeros(nq, 64, dtype=torch.float32, device="cuda")
    out = C.csa2_sparse_attn_decode(cache, bf16_dev(q), bf16_dev(swa), torch.from_numpy(idx).cuda(),
                                    float(SCALE), swa_len=torch.from_numpy(swa_len).cuda(), lse=lse)
    out = bf16_host(out)
    lse = lse.cpu().numpy()
    for i in range(nq):
        codes, scales = O.quantise(ents[i], layout)
        _, o, ol = O.sparse_attention(q[i], codes, scales, layout, idx[i], swa[i, :swa_len[i]],
                                      SCALE)
        check_attn(out[i], o)
        check_lse(lse[i], ol)
    assert cache.device_error() == 0


def test_sharper_softmax_and_reuse_identity(C):
    """A larger scale concentrates the weights (exercises the running-max
    rescale); a Reuse layer with the Full layer's indices, q and window
    reproduces its output bit for bit."""
    import torch
    rng = np.random.default_rng(5)
    cache, ents = _cache(C, [4000, 4000], 4096, 33)
    q = S.normal_bf16(S.stream_key(34, S.S_Q, 0), 0, 2 * 64 * 512).reshape(2, 64, 512)
    swa = S.normal_bf16(S.stream_key(34, S.S_SWA, 0), 0, 2 * 128 * 512).reshape(2, 128, 512)
    idx = np.stack([_sel(rng, 4000), _sel(rng, 4000)])
    ti = torch.from_numpy(idx).cuda()
    for scale in (np.float32(0.25), np.float32(0.01)):
        a = C.csa2_sparse_attn_decode(cache, bf16_dev(q), bf16_dev(swa), ti, float(scale))
        b = C.csa2_sparse_attn_decode(cache, bf16_dev(q), bf16_dev(swa), ti, float(scale))
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        out = bf16_host(a)
        for i in range(2):
            codes, scales = O.quantise(ents[i], 0)
            _, o, _ = O.sparse_attention(q[i], codes, scales, 0, idx[i], swa[i], scale)
            check_attn(out[i], o)


def test_empty_candidates_and_bad_index(C):
    import torch
    cache, ents = _cache(C, [10, 10], 64, 35)
    q = S.normal_bf16(S.stream_key(36, S.S_Q, 0), 0, 2 * 64 * 512).reshape(2, 64, 512)
    swa = S.normal_bf16(S.stream_key(36, S.S_SWA, 0), 0, 2 * 128 * 512).reshape(2, 128, 512)
    idx = np.full((2, 512), -1, np.int32)
    idx[1, :3] = [2, 9, 10]                # 10 is out of range: skipped and reported
    lse = torch.zeros(2, 64, device="cuda")
    out = C.csa2_sparse_attn_decode(cache, bf16_dev(q), bf16_dev(swa), torch.from_numpy(idx).cuda(),
                                    float(SCALE), swa_len=torch.tensor([0, 5], dtype=torch.int32,
                                                                       device="cuda"), lse=lse)
    o = bf16_host(out)
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0].cpu().numpy()))
    codes, scales = O.quantise(ents[1], 0)
    _, ref, _ = O.sparse_attention(q[1], codes, scales, 0, np.array([2, 9], np.int32),
                                   swa[1, :5], SCALE)
    check_attn(o[1], ref)
    assert cache.device_error() == 7
    assert cache.device_error() == 0       # reading clears the word


@pytest.mark.parametrize("ratio", [1, 2])
def test_prefill_window_band(C, ratio):
    import torch
    rng = np.random.default_rng(ratio)
    n_ent = 800
    cache, ents = _cache(C, [n_ent], 1024, 37, ratio=ratio)
    nq, pos0 = 20, 1500 if ratio == 2 else 700
    swa_pos0 = pos0 - 60                   # a replay that starts 60 tokens back
    rows = S.normal_bf16(S.stream_key(38, S.S_SWA, 1), 0, (nq + 60) * 512).reshape(nq + 60, 512)
    q = S.normal_bf16(S.stream_key(38, S.S_Q, 1), 0, nq * 64 * 512).reshape(nq, 64, 512)
    idx = np.stack([_sel(rng, O.visible_entries(n_ent, ratio, pos0 + i)) for i in range(nq)])
    out = C.csa2_sparse_attn_prefill(cache, 0, pos0, bf16_dev(q), bf16_dev(rows), swa_pos0,
                                     torch.from_numpy(idx).cuda(), float(SCALE))
    out = bf16_host(out)
    codes, scales = O.quantise(ents[0], 0)
    for i in range(nq):
        lo, hi = O.swa_rows(pos0 + i, 128, swa_pos0)
        _, o, _ = O.sparse_attention(q[i], codes, scales, 0, idx[i],
                                     rows[lo - swa_pos0:hi - swa_pos0], SCALE)
        check_attn(out[i], o)


@pytest.mark.parametrize("n_q", [3, 50, 200])
def test_split_and_single_cta_paths_agree_with_oracle(C, n_q):
    """With a workspace, a small batch (3 or 50 queries) splits each query's
    candidate tiles over two CTAs and merges their softmax states; without
    one (or for a large batch: 200 queries) one CTA takes every tile.  Both
    match the oracle."""
    import torch
    rng = np.random.default_rng(n_q)
    lens = [int(x) for x in rng.integers(100, 3000, n_q)]
    cache, ents = _cache(C, lens, 3072, 51)
    q = S.normal_bf16(S.stream_key(52, S.S_Q, 0), 0, n_q * 64 * 512).reshape(n_q, 64, 512)
    swa = S.normal_bf16(S.stream_key(52, S.S_SWA, 0), 0, n_q * 128 * 512).reshape(n_q, 128, 512)
    idx = np.stack([_sel(rng, n) for n in lens])
    swa_len = torch.from_numpy(rng.integers(0, 129, n_q).astype(np.int32)).cuda()
    outs = []
    for ws in (None, torch.empty(0, dtype=torch.uint8, device="cuda")):
        lse = torch.zeros(n_q, 64, device="cuda")
        o = C.csa2_sparse_attn_decode(cache, bf16_dev(q), bf16_dev(swa), torch.from_numpy(idx).cuda(),
                                      float(SCALE), swa_len=swa_len, lse=lse, workspace=ws)
        outs.append((bf16_host(o), lse.cpu().numpy()))
    sl = swa_len.cpu().numpy()
    for i in range(0, n_q, max(1, n_q // 7)):
        codes, scales = O.quantise(ents[i], 0)
        _, ref, rl = O.sparse_attention(q[i], codes, scales, 0, idx[i], swa[i, :sl[i]], SCALE)
        for o, l in outs:
            check_attn(o[i], ref)
            assert np.allclose(l[i], rl, atol=1e-3, rtol=0)
    assert cache.device_error() == 0



def _aligned_cache(C, gains, seed=53):
    """4096 entries in four ranges of 1024; range j is N(0, 1/16) noise plus
    gains[j] / 2 times the query of head (s mod 64), so that head's logits in
    the top-k tile drawn from range j grow with gains[j] (read with twice
    the usual softmax scale, values stay below about 2 in magnitude)."""
    n = 4096
    q = S.normal_bf16(S.stream_key(seed + 2, S.S_Q, 0), 0, 64 * 512).reshape(64, 512)
    qf = S.bf16_bits_to_f32(q)
    e = S.normal_f32(S.stream_key(seed, S.S_ENTRIES, 0), 0, n * 512).reshape(n, 512)
    for j, gain in enumerate(gains):
        rows = np.arange(j * 1024, (j + 1) * 1024)
        e[rows] = e[rows] * np.float32(0.25) + np.float32(gain / 2) * qf[rows % 64]
    cache = C.Cache(C.config(), [n])
    k = S.normal_bf16(S.stream_key(seed, S.S_IDXK, 0), 0, n * 128).reshape(n, 128)
    C.csa2_append_entries(cache, [0], [n], f32_dev(e), bf16_dev(k))
    rng = np.random.default_rng(seed + 1)
    idx = np.concatenate([np.sort(rng.choice(1024, 128, replace=False)) + 1024 * j
                          for j in range(4)]).astype(np.int32)[None]
    swa = S.normal_bf16(S.stream_key(seed + 2, S.S_SWA, 0), 0, 128 * 512).reshape(1, 128, 512)
    return cache, e, q[None], swa, idx


@pytest.mark.parametrize("gains", [(0.0, 0.2, 0.35, 1.0), (1.0, 0.35, 0.2, 0.0)])
def test_running_max_moves_and_stays(C, gains):
    """Each head's logits jump tile after tile (its running maximum moves by
    more than 2^8 at the fully aligned tile and by less at the partly aligned
    ones), or jump once and fall back: the split and single-CTA paths both
    match the oracle."""
    import torch
    cache, e, q, swa, idx = _aligned_cache(C, gains)
    scale = np.float32(2 * SCALE)
    codes, scales = O.quantise(e, 0)
    _, ref, rl = O.sparse_attention(q[0], codes, scales, 0, idx[0], swa[0], scale)
    for ws in (None, torch.empty(0, dtype=torch.uint8, device="cuda")):
        lse = torch.zeros(1, 64, device="cuda")
        out = C.csa2_sparse_attn_decode(cache, bf16_dev(q), bf16_dev(swa),
                                        torch.from_numpy(idx).cuda(), float(scale), lse=lse,
                                        workspace=ws)
        check_attn(bf16_host(out)[0], ref)
        assert np.allclose(lse.cpu().numpy()[0], rl, atol=1e-3 * max(1.0, np.abs(rl).max()),
                           rtol=0)
    assert cache.device_error() == 0


def test_large_values_stay_within_the_probability_rounding_bound(C):
    """Entries eight times larger everywhere: the probabilities that weight
    the values are rounded to bf16 for the tensor cores (relative error at
    most 2^-9, twice over when the running maximum is not the final one), so
    where large values cancel, an output's error scales with sum_j p_j |kv_j|
    rather than with |o|.  The bound derived from that arithmetic,
    2^-8 (sum_j p_j |kv_j| + |o|), holds element by element."""
    import torch
    n = 4096
    cache = C.Cache(C.config(), [n])
    e = S.normal_f32(S.stream_key(53, S.S_ENTRIES, 0), 0, n * 512).reshape(n, 512) * 8
    k = S.normal_bf16(S.stream_key(53, S.S_IDXK, 0), 0, n * 128).reshape(n, 128)
    C.csa2_append_entries(cache, [0], [n], f32_dev(e), bf16_dev(k))
    rng = np.random.default_rng(54)
    idx = np.concatenate([np.sort(rng.choice(1024, 128, replace=False)) + 1024 * j
                          for j in range(4)]).astype(np.int32)[None]
    q = S.normal_bf16(S.stream_key(55, S.S_Q, 0), 0, 64 * 512).reshape(1, 64, 512)
    swa = S.normal_bf16(S.stream_key(55, S.S_SWA, 0), 0, 128 * 512).reshape(1, 128, 512)
    codes, scales = O.quantise(e, 0)
    _, ref, _ = O.sparse_attention(q[0], codes, scales, 0, idx[0], swa[0], SCALE)
    kv = np.concatenate([S.bf16_bits_to_f32(swa[0]).astype(np.float64),
                         O.dequantise(codes, scales, 0)[idx[0]].astype(np.float64)])
    logit = (S.bf16_bits_to_f32(q[0]).astype(np.float64) @ kv.T) * float(SCALE)
    pw = np.exp(logit - logit.max(1, keepdims=True))
    pw /= pw.sum(1, keepdims=True)
    bound = 2.0 ** -8 * (pw @ np.abs(kv) + np.abs(ref))
    for ws in (None, torch.empty(0, dtype=torch.uint8, device="cuda")):
        out = C.csa2_sparse_attn_decode(cache, bf16_dev(q), bf16_dev(swa),
                                        torch.from_numpy(idx).cuda(), float(SCALE), workspace=ws)
        g = S.bf16_bits_to_f32(bf16_host(out)[0]).astype(np.float64)
        assert np.all(np.abs(g - ref) <= bound), float((np.abs(g - ref) / bound).max())
    assert cache.device_error() == 0


@pytest.mark.parametrize("split", [False, True])
def test_layers_in_one_launch_equal_separate_calls(C, split):
    """csa2_sparse_attn_decode_layers: four layers of a group (own queries,
    windows, outputs; one selection) in one launch give, layer by layer,
    exactly the outputs and lse of separate csa2_sparse_attn_decode calls,
    with and without the two-CTA split; layer 2 checked against the
    oracle."""
    import torch
    rng = np.random.default_rng(71)
    lens = [900, 2000, 3000]
    cache, ents = _cache(C, lens, 3072, 72)
    nq, L = len(lens), 4
    qs = [S.normal_bf16(S.stream_key(73, S.S_Q, l), 0, nq * 64 * 512).reshape(nq, 64, 512)
          for l in range(L)]
    swas = [S.normal_bf16(S.stream_key(73, S.S_SWA, l), 0, nq * 128 * 512).reshape(nq, 128, 512)
            for l in range(L)]
    swa_len = torch.tensor([128, 7, 64], dtype=torch.int32, device="cuda")
    idx = np.stack([_sel(rng, n) for n in lens])
    idx_d = torch.from_numpy(idx).cuda()
    ws = None if split else torch.empty(0, dtype=torch.uint8, device="cuda")
    q_d = [bf16_dev(x) for x in qs]
    s_d = [bf16_dev(x) for x in swas]
    outs = [torch.empty(nq, 64, 512, dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    lses = [torch.empty(nq, 64, device="cuda") for _ in range(L)]
    C.csa2_sparse_attn_decode_layers(cache, q_d, s_d, idx_d, float(SCALE), outs, lses,
                                     swa_len=swa_len, workspace=ws)
    for l in range(L):
        lse1 = torch.empty(nq, 64, device="cuda")
        o1 = C.csa2_sparse_attn_decode(cache, q_d[l], s_d[l], idx_d, float(SCALE),
                                       swa_len=swa_len, lse=lse1, workspace=ws)
        assert torch.equal(o1.view(torch.int16), outs[l].view(torch.int16)), l
        assert torch.equal(lse1, lses[l]), l
    o = bf16_host(outs[2])
    ln = swa_len.cpu().numpy()
    for i in range(nq):
        codes, scales = O.quantise(ents[i], 0)
        _, ref, rl = O.sparse_attention(qs[2][i], codes, scales, 0, idx[i], swas[2][i, :ln[i]], SCALE)
        check_attn(o[i], ref)
        check_lse(lses[2].cpu().numpy()[i], rl)
    assert cache.device_error() == 0


@pytest.mark.parametrize("ratio,fp8", [(1, False), (2, False), (2, True)])
def test_prefill_layers_in_one_launch_equal_separate_calls(C, ratio, fp8):
    """csa2_sparse_attn_prefill_layers: three layers of a chunk (own queries,
    window rows -- bf16 or FP8 --, sinks and outputs; one selection; output
    RoPE on) in one launch give, layer by layer, exactly the outputs and lse
    of separate csa2_sparse_attn_prefill calls; layer 1 checked against the
    oracle."""
    import torch
    rng = np.random.default_rng(91 + ratio + 10 * fp8)
    n_ent = 900
    cache, ents = _cache(C, [n_ent], 1024, 92, ratio=ratio)
    nq, pos0, L = 30, 1700 if ratio == 2 else 850, 3
    swa_pos0 = pos0 - 50
    rows = [S.normal_bf16(S.stream_key(93, S.S_SWA, l), 0, (nq + 50) * 512).reshape(nq + 50, 512)
            for l in range(L)]
    qs = [S.normal_bf16(S.stream_key(93, S.S_Q, l), 0, nq * 64 * 512).reshape(nq, 64, 512)
          for l in range(L)]
    sinks = [rng.standard_normal(64).astype(np.float32) for _ in range(L)]
    idx = np.stack([_sel(rng, O.visible_entries(n_ent, ratio, pos0 + i)) for i in range(nq)])
    idx_d = torch.from_numpy(idx).cuda()
    q_d, r_d, s_d = [bf16_dev(x) for x in qs], [bf16_dev(x) for x in rows], [f32_dev(x) for x in sinks]
    outs = [torch.empty(nq, 64, 512, dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    lses = [torch.empty(nq, 64, device="cuda") for _ in range(L)]
    f8 = [C.csa2_swa_fp8_quantise(x) for x in r_d] if fp8 else None
    C.csa2_sparse_attn_prefill_layers(cache, 0, pos0, q_d, None if fp8 else r_d, swa_pos0, idx_d,
                                      float(SCALE), outs, lses, sinks=s_d, rope_out=True,
                                      rope_base=5e5, swa_fp8s=f8)
    for l in range(L):
        lse1 = torch.empty(nq, 64, device="cuda")
        o1 = C.csa2_sparse_attn_prefill(cache, 0, pos0, q_d[l], None if fp8 else r_d[l], swa_pos0,
                                        idx_d, float(SCALE), lse=lse1, sink=s_d[l], rope_out=True,
                                        rope_base=5e5, swa_fp8=f8[l] if fp8 else None)
        assert torch.equal(o1.view(torch.int16), outs[l].view(torch.int16)), l
        assert torch.equal(lse1, lses[l]), l
    out = bf16_host(outs[1])
    lse = lses[1].cpu().numpy()
    codes, scales = O.quantise(ents[0], 0)
    for i in range(0, nq, 3):
        lo, hi = O.swa_rows(pos0 + i, 128, swa_pos0)
        win = rows[1][lo - swa_pos0:hi - swa_pos0]
        if fp8:
            win = O.swa_fp8_round_bf16(win)
        _, o, ol = O.sparse_attention(qs[1][i], codes, scales, 0, idx[i], win, SCALE)
        _, o2, ol2 = O.attention_epilogue(o, ol, sink=sinks[1], rope_pos=pos0 + i, rope_base=5e5)
        check_attn(out[i], o2)
        check_lse(lse[i], ol2)
    assert cache.device_error() == 0


def test_layers_epilogue_options_per_layer(C):
    """Per-layer sinks and FP8 window rows in one launch equal the separate
    calls with the same options; the output RoPE must be one setting for
    the launch."""
    import torch
    rng = np.random.default_rng(81)
    lens = [1500, 600]
    cache, _ = _cache(C, lens, 1536, 82)
    nq, L = len(lens), 3
    qs = [bf16_dev(S.normal_bf16(S.stream_key(83, S.S_Q, l), 0, nq * 64 * 512).reshape(nq, 64, 512))
          for l in range(L)]
    rows = [bf16_dev(S.normal_bf16(S.stream_key(83, S.S_SWA, l), 0, nq * 128 * 512).reshape(nq * 128, 512))
            for l in range(L)]
    f8 = [C.csa2_swa_fp8_quantise(r) for r in rows]
    sinks = [torch.linspace(-1.0 - l, 1.0 + l, 64, device="cuda") for l in range(L)]
    pos = torch.tensor([4000, 123456], dtype=torch.int64, device="cuda")
    idx_d = torch.from_numpy(np.stack([_sel(rng, n) for n in lens])).cuda()
    outs = [torch.empty(nq, 64, 512, dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    lses = [torch.empty(nq, 64, device="cuda") for _ in range(L)]
    C.csa2_sparse_attn_decode_layers(cache, qs, [None] * L, idx_d, float(SCALE), outs, lses,
                                     sinks=sinks, rope_pos=pos, swa_fp8s=f8)
    for l in range(L):
        lse1 = torch.empty(nq, 64, device="cuda")
        o1 = C.csa2_sparse_attn_decode(cache, qs[l], None, idx_d, float(SCALE), lse=lse1,
                                       sink=sinks[l], rope_pos=pos, swa_fp8=f8[l])
        assert torch.equal(o1.view(torch.int16), outs[l].view(torch.int16)), l
        assert torch.equal(lse1, lses[l]), l
    # RoPE on some layers only: refused before any launch
    with pytest.raises(C.Csa2Error, match="INVALID_ARG"):
        opts = [C.AttnOpts(None, C._ptr(pos), 1, 0.0, None, None, None),
                C.AttnOpts(None, None, 0, 0.0, None, None, None)]
        import ctypes
        arr = lambda xs: (ctypes.c_void_p * 2)(*[C._ptr(x) for x in xs])
        oarr = (ctypes.c_void_p * 2)(*[ctypes.cast(ctypes.pointer(o), ctypes.c_void_p) for o in opts])
        C._check(C.lib.csa2_sparse_attn_decode_layers(
            cache.handle, 2, nq, None, arr(qs[:2]), arr(rows[:2]), None, C._ptr(idx_d),
            float(SCALE), arr(outs[:2]), None, None, 0, oarr, C._stream(None)), "layers")
    assert cache.device_error() == 0


@pytest.mark.parametrize("fp8", [False, True])
def test_batch_equals_chunked_launches(C, fp8):
    """A readout launch of more (query, layer) items than SMs gives, bit for
    bit, the outputs and lse of launches over chunks of its queries, over
    queries with no entry and no window row (no tile at all), short and full
    windows, bf16 or FP8 window rows; a sample of queries is checked against
    the oracle."""
    import torch
    rng = np.random.default_rng(101 + fp8)
    nq, L = 170, 2
    lens = [int(x) for x in rng.integers(0, 1200, nq)]
    for i in range(0, nq, 17):
        lens[i] = 0
    cache, ents = _cache(C, lens, 1200, 102)
    swl = rng.integers(0, 129, nq).astype(np.int32)
    swl[::17] = 0                            # with lens[i] = 0: no tile
    swl[5::17] = 128
    qs = [S.normal_bf16(S.stream_key(103, S.S_Q, l), 0, nq * 64 * 512).reshape(nq, 64, 512)
          for l in range(L)]
    swas = [S.normal_bf16(S.stream_key(103, S.S_SWA, l), 0, nq * 128 * 512).reshape(nq, 128, 512)
            for l in range(L)]
    idx = np.stack([_sel(rng, n) for n in lens])
    idx_d = torch.from_numpy(idx).cuda()
    q_d = [bf16_dev(x) for x in qs]
    s_d = [bf16_dev(x) for x in swas]
    f8 = [C.csa2_swa_fp8_quantise(x) for x in s_d] if fp8 else None
    swl_d = torch.from_numpy(swl).cuda()
    no_split = torch.empty(0, dtype=torch.uint8, device="cuda")

    def run(lo, hi):
        outs = [torch.empty(hi - lo, 64, 512, dtype=torch.bfloat16, device="cuda") for _ in range(L)]
        lses = [torch.empty(hi - lo, 64, device="cuda") for _ in range(L)]
        f8s = None if f8 is None else [tuple(t[lo * 128:hi * 128] for t in f) for f in f8]
        C.csa2_sparse_attn_decode_layers(
            cache, [x[lo:hi] for x in q_d], None if fp8 else [x[lo:hi] for x in s_d],
            idx_d[lo:hi], float(SCALE), outs, lses, swa_len=swl_d[lo:hi],
            seq_ids=list(range(lo, hi)), workspace=no_split, swa_fp8s=f8s)
        return outs, lses

    outs, lses = run(0, nq)
    for lo in range(0, nq, 30):
        hi = min(nq, lo + 30)
        o1, l1 = run(lo, hi)
        for l in range(L):
            assert torch.equal(o1[l].view(torch.int16), outs[l][lo:hi].view(torch.int16)), (lo, l)
            assert torch.equal(l1[l], lses[l][lo:hi]), (lo, l)
    o = bf16_host(outs[1])
    ls = lses[1].cpu().numpy()
    for i in (0, 5, 22, 100, 169):
        if lens[i] == 0 and swl[i] == 0:
            assert np.all(o[i] == 0) and np.all(np.isneginf(ls[i]))
            continue
        rows = swas[1][i, :swl[i]]
        if fp8:
            rows = O.swa_fp8_round_bf16(rows)
        codes, scales = O.quantise(ents[i], 0)
        _, ref, rl = O.sparse_attention(qs[1][i], codes, scales, 0, idx[i], rows, SCALE)
        check_attn(o[i], ref)
        check_lse(ls[i], rl)
    assert cache.device_error() == 0
