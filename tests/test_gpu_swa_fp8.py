"""FP8 window rows ("DeepSeek-V4.1-Flash" report, section 2.4.4: the SWA KV
cache stays FP8) against the oracle: the quantisation bit-exact, and the
readout over FP8 window rows equal (same bar as the plain readout) to the
oracle's attention over the rows taken through FP8 and back, on decode
(split and single-CTA paths, both main-KV layouts, partial windows) and
prefill, alone and with the sink / output-RoPE options."""
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


def test_quantisation_is_the_oracles(C):
    import torch
    rng = np.random.default_rng(130)
    n = 777
    x = rng.standard_normal((n, 512)) * np.exp(rng.uniform(-20, 20, (n, 1)))
    x[3] = 0.0                                   # an all-zero row
    x[4, :64] = -0.0
    x[5, 100] = 1e30                             # a block dominated by one value
    bits = S.f32_to_bf16_bits(x.astype(np.float32))
    codes, rope, scales = C.csa2_swa_fp8_quantise(bf16_dev(bits))
    oc, orp, osc = O.swa_fp8_quantise(bits)
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(scales.cpu().numpy(), osc)
    assert np.array_equal(bf16_host(rope), orp)


@pytest.mark.parametrize("layout", [0, 1])
def test_decode_over_fp8_window(C, layout):
    import torch
    rng = np.random.default_rng(131 + layout)
    lens = [3000, 700, 5000]
    cache, ents = _cache(C, lens, 5120, 132, layout)
    nq = len(lens)
    q = S.normal_bf16(S.stream_key(133, S.S_Q, 0), 0, nq * 64 * 512).reshape(nq, 64, 512)
    swa = S.normal_f32(S.stream_key(133, S.S_SWA, 0), 0, nq * 128 * 512).reshape(nq, 128, 512)
    swa[:, :, 200] *= 8                          # an outlier channel
    swa = S.f32_to_bf16_bits(swa)
    swa_len = np.array([128, 37, 0], np.int32)
    idx = np.stack([_sel(rng, n) for n in lens])
    f8 = C.csa2_swa_fp8_quantise(bf16_dev(swa))
    for ws in (None, torch.empty(0, dtype=torch.uint8, device="cuda")):
        lse = torch.zeros(nq, 64, device="cuda")
        out = C.csa2_sparse_attn_decode(cache, bf16_dev(q), None, torch.from_numpy(idx).cuda(),
                                        float(SCALE), swa_len=torch.from_numpy(swa_len).cuda(),
                                        lse=lse, workspace=ws, swa_fp8=f8)
        out = bf16_host(out)
        lse = lse.cpu().numpy()
        for i in range(nq):
            codes, scales = O.quantise(ents[i], layout)
            rows = O.swa_fp8_round_bf16(swa[i, :swa_len[i]])
            _, o, ol = O.sparse_attention(q[i], codes, scales, layout, idx[i], rows, SCALE)
            check_attn(out[i], o)
            check_lse(lse[i], ol)
    assert cache.device_error() == 0


@pytest.mark.parametrize("ratio", [1, 2])
def test_prefill_over_fp8_window_with_sink_and_rope(C, ratio):
    import torch
    rng = np.random.default_rng(134 + ratio)
    n_ent = 900
    cache, ents = _cache(C, [n_ent], 1024, 136, ratio=ratio)
    nq, pos0 = 20, 1700 if ratio == 2 else 850
    swa_pos0 = pos0 - 50
    rows = S.normal_bf16(S.stream_key(137, S.S_SWA, 1), 0, (nq + 50) * 512).reshape(nq + 50, 512)
    q = S.normal_bf16(S.stream_key(137, S.S_Q, 1), 0, nq * 64 * 512).reshape(nq, 64, 512)
    idx = np.stack([_sel(rng, O.visible_entries(n_ent, ratio, pos0 + i)) for i in range(nq)])
    sink = rng.standard_normal(64).astype(np.float32)
    f8 = C.csa2_swa_fp8_quantise(bf16_dev(rows))
    out = C.csa2_sparse_attn_prefill(cache, 0, pos0, bf16_dev(q), None, swa_pos0,
                                     torch.from_numpy(idx).cuda(), float(SCALE),
                                     sink=f32_dev(sink), rope_out=True, swa_fp8=f8)
    out = bf16_host(out)
    rows8 = O.swa_fp8_round_bf16(rows)
    codes, scales = O.quantise(ents[0], 0)
    for i in range(nq):
        lo, hi = O.swa_rows(pos0 + i, 128, swa_pos0)
        _, o, ol = O.sparse_attention(q[i], codes, scales, 0, idx[i],
                                      rows8[lo - swa_pos0:hi - swa_pos0], SCALE)
        _, o2, _ = O.attention_epilogue(o, ol, sink=sink, rope_pos=pos0 + i)
        check_attn(out[i], o2)
    assert cache.device_error() == 0


def test_fp8_options_must_come_together(C):
    import ctypes
    import torch
    cache, _ = _cache(C, [100], 128, 138)
    q = torch.zeros(1, 64, 512, dtype=torch.bfloat16, device="cuda")
    ti = torch.full((1, 512), -1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    codes = torch.zeros(128, 448, dtype=torch.uint8, device="cuda")
    opts = C.AttnOpts(None, None, 0, 0.0, codes.data_ptr(), None, None)
    st = C.lib.csa2_sparse_attn_decode_ex(cache.handle, 1, None, q.data_ptr(), None, None,
                                          ti.data_ptr(), ctypes.c_float(0.1), out.data_ptr(),
                                          None, None, 0, ctypes.byref(opts), None)
    assert st == 1      # CSA2_ERR_INVALID_ARG
