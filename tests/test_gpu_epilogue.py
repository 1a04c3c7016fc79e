"""GPU readout epilogue variants ("DeepSeek-V4" blog reading, section 4.3):
attention sink and output RoPE(-i), against the oracle's epilogue applied
to its fp64 attention, on the decode (split and single-CTA) and prefill
paths; the same parity bar as the plain readout."""
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


def _cache(C, lens, cap, seed, layout=0, ratio=1):
    cache = C.Cache(C.config(layout=layout, ratio=ratio), [cap] * len(lens))
    ents = []
    for s, n in enumerate(lens):
        e = S.normal_f32(S.stream_key(seed, S.S_ENTRIES, s), 0, n * 512).reshape(n, 512)
        k = S.normal_bf16(S.stream_key(seed, S.S_IDXK, s), 0, n * 128).reshape(n, 128)
        if n:
            C.csa2_append_entries(cache, [s], [n], f32_dev(e), bf16_dev(k))
        ents.append(e)
    return cache, ents


def _sel(rng, n, k=512):
    m = min(n, k)
    out = np.full(k, -1, np.int32)
    out[:m] = np.sort(rng.choice(n, m, replace=False))
    return out


@pytest.mark.parametrize("layout", [0, 1])
def test_decode_sink_and_rope(C, layout):
    import torch
    rng = np.random.default_rng(70 + layout)
    lens = [3000, 600, 5000, 40]
    cache, ents = _cache(C, lens, 5120, 71, layout)
    nq = len(lens)
    q = S.normal_bf16(S.stream_key(72, S.S_Q, 0), 0, nq * 64 * 512).reshape(nq, 64, 512)
    swa = S.normal_bf16(S.stream_key(72, S.S_SWA, 0), 0, nq * 128 * 512).reshape(nq, 128, 512)
    swa_len = np.array([128, 7, 0, 0], np.int32)
    idx = np.stack([_sel(rng, n) for n in lens])
    idx[3, :] = -1                                  # query 3: nothing at all
    sink = (rng.standard_normal(64) * 2).astype(np.float32)
    sink[5] = -np.inf                               # a head without sink
    sink[9] = 40.0                                  # a sink that swallows the head
    pos = np.array([2999, 1 << 20, 0, 123456], np.int64)
    for ws in (None, torch.empty(0, dtype=torch.uint8, device="cuda")):
        lse = torch.zeros(nq, 64, device="cuda")
        out = C.csa2_sparse_attn_decode(cache, bf16_dev(q), bf16_dev(swa),
                                        torch.from_numpy(idx).cuda(), float(SCALE),
                                        swa_len=torch.from_numpy(swa_len).cuda(), lse=lse,
                                        workspace=ws, sink=f32_dev(sink),
                                        rope_pos=torch.from_numpy(pos).cuda())
        out = bf16_host(out)
        lse = lse.cpu().numpy()
        for i in range(nq):
            codes, scales = O.quantise(ents[i], layout)
            _, o, ol = O.sparse_attention(q[i], codes, scales, layout, idx[i],
                                          swa[i, :swa_len[i]], SCALE)
            _, o2, ol2 = O.attention_epilogue(o, ol, sink=sink, rope_pos=int(pos[i]))
            check_attn(out[i], o2)
            fin = np.isfinite(ol2)
            assert np.array_equal(np.isfinite(lse[i]), fin)
            check_lse(lse[i][fin], ol2[fin])
    assert cache.device_error() == 0


def test_neutral_options_leave_the_output_unchanged(C):
    """A sink of -inf on every head and RoPE at position 0 give the plain
    readout (as values)."""
    import torch
    rng = np.random.default_rng(73)
    cache, _ = _cache(C, [2000, 2000], 2048, 74)
    q = S.normal_bf16(S.stream_key(75, S.S_Q, 0), 0, 2 * 64 * 512).reshape(2, 64, 512)
    swa = S.normal_bf16(S.stream_key(75, S.S_SWA, 0), 0, 2 * 128 * 512).reshape(2, 128, 512)
    ti = torch.from_numpy(np.stack([_sel(rng, 2000), _sel(rng, 2000)])).cuda()
    plain = C.csa2_sparse_attn_decode(cache, bf16_dev(q), bf16_dev(swa), ti, float(SCALE))
    neutral = C.csa2_sparse_attn_decode(cache, bf16_dev(q), bf16_dev(swa), ti, float(SCALE),
                                        sink=torch.full((64,), -float("inf"), device="cuda"),
                                        rope_pos=torch.zeros(2, dtype=torch.int64, device="cuda"))
    assert torch.equal(plain.float(), neutral.float())


@pytest.mark.parametrize("ratio", [1, 2])
def test_prefill_sink_and_rope(C, ratio):
    import torch
    rng = np.random.default_rng(76 + ratio)
    n_ent = 900
    cache, ents = _cache(C, [n_ent], 1024, 78, ratio=ratio)
    nq, pos0 = 24, 1700 if ratio == 2 else 850
    swa_pos0 = pos0 - 40
    rows = S.normal_bf16(S.stream_key(79, S.S_SWA, 1), 0, (nq + 40) * 512).reshape(nq + 40, 512)
    q = S.normal_bf16(S.stream_key(79, S.S_Q, 1), 0, nq * 64 * 512).reshape(nq, 64, 512)
    idx = np.stack([_sel(rng, O.visible_entries(n_ent, ratio, pos0 + i)) for i in range(nq)])
    sink = rng.standard_normal(64).astype(np.float32)
    lse = torch.zeros(nq, 64, device="cuda")
    out = C.csa2_sparse_attn_prefill(cache, 0, pos0, bf16_dev(q), bf16_dev(rows), swa_pos0,
                                     torch.from_numpy(idx).cuda(), float(SCALE), lse=lse,
                                     sink=f32_dev(sink), rope_out=True, rope_base=5e5)
    out = bf16_host(out)
    lse = lse.cpu().numpy()
    codes, scales = O.quantise(ents[0], 0)
    for i in range(nq):
        lo, hi = O.swa_rows(pos0 + i, 128, swa_pos0)
        _, o, ol = O.sparse_attention(q[i], codes, scales, 0, idx[i],
                                      rows[lo - swa_pos0:hi - swa_pos0], SCALE)
        _, o2, ol2 = O.attention_epilogue(o, ol, sink=sink, rope_pos=pos0 + i, rope_base=5e5)
        check_attn(out[i], o2)
        check_lse(lse[i], ol2)
    assert cache.device_error() == 0


def test_rope_needs_positions_in_decode(C):
    import ctypes
    import torch
    cache, _ = _cache(C, [100], 128, 80)
    q = torch.zeros(1, 64, 512, dtype=torch.bfloat16, device="cuda")
    swa = torch.zeros(1, 128, 512, dtype=torch.bfloat16, device="cuda")
    ti = torch.full((1, 512), -1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    opts = C.AttnOpts(None, None, 1, 0.0)
    st = C.lib.csa2_sparse_attn_decode_ex(cache.handle, 1, None, q.data_ptr(), swa.data_ptr(),
                                          None, ti.data_ptr(), ctypes.c_float(0.1),
                                          out.data_ptr(), None, None, 0, ctypes.byref(opts),
                                          None)
    assert st == 1      # CSA2_ERR_INVALID_ARG, nothing launched
