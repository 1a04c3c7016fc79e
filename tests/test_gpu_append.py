"""GPU parity of the compressor and the FP4 quantise-append against the
oracle: bit-exact codes, scales, compressed values and indexer keys."""
import numpy as np
import pytest

import csa2_synth as S
import oracle as O
from tests._parity import bf16_dev, bf16_host, f32_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def C():
    import fp4_kv_cache_index_gb300 as C
    return C


def _codec_rows(layout):
    """Blocks that walk every scale byte (and the ties between E4M3 values),
    every E2M1 code, extreme and signed-zero values, then random rows."""
    rows = []
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], np.float32)
    g = O.group(layout)
    if layout == 0:
        scales = [O.ue8m0_value(b) for b in range(0, 253)]   # 6 * scale stays finite
    else:
        vals = [O.e4m3_value(b) for b in range(0, 0x7F)]
        mids = [(a + b) / 2 for a, b in zip(vals, vals[1:])]
        scales = vals + mids + [449.0, 500.0, 1e6]
    for s in scales:
        r = np.zeros(512, np.float32)
        for b in range(512 // g):
            blk = np.zeros(g, np.float32)
            blk[0] = np.float32(6.0 * s)
            blk[1:9] = grid * np.float32(s)
            blk[9:17 if g > 16 else g] = -grid[:len(blk[9:17 if g > 16 else g])] * np.float32(s)
            if g > 16:
                blk[17:] = np.float32(s) * np.linspace(-7, 7, g - 17, dtype=np.float32)
            r[b * g:(b + 1) * g] = np.roll(blk, b)
        rows.append(r)
    special = np.zeros((4, 512), np.float32)
    special[1] = -0.0
    special[2, ::7] = 1e-42
    special[3] = np.float32(3e38) * np.sign(np.linspace(-1, 1, 512, dtype=np.float32))
    rows.extend(special)
    rng = np.random.default_rng(layout)
    mag = 10.0 ** rng.uniform(-30, 5, (20000, 1))
    rows.extend((rng.standard_normal((20000, 512)) * mag).astype(np.float32))
    return np.stack(rows).astype(np.float32)


@pytest.mark.parametrize("layout", [0, 1])
def test_append_entries_bit_exact(C, layout):
    x = _codec_rows(layout)
    n = x.shape[0]
    kx = S.normal_bf16(S.stream_key(7, S.S_IDXK, 0), 0, n * 128).reshape(n, 128)
    cache = C.Cache(C.config(layout=layout), [n // 2 + 10, n - n // 2])
    h = n // 2
    # two sequences in one call, then a second call onto sequence 0
    C.csa2_append_entries(cache, [1, 0], [n - h, h - 5], f32_dev(np.concatenate([x[h:], x[:h - 5]])),
                          bf16_dev(np.concatenate([kx[h:], kx[:h - 5]])))
    C.csa2_append_entries(cache, [0], [5], f32_dev(x[h - 5:h]), bf16_dev(kx[h - 5:h]))
    v = cache.views()
    off = v["entry_offset"]
    codes = np.concatenate([v["codes"][off[0]:off[0] + h].cpu().numpy(),
                            v["codes"][off[1]:off[1] + n - h].cpu().numpy()])
    scales = np.concatenate([v["scales"][off[0]:off[0] + h].cpu().numpy(),
                             v["scales"][off[1]:off[1] + n - h].cpu().numpy()])
    ik = np.concatenate([bf16_host(v["idx_k"][off[0]:off[0] + h]),
                         bf16_host(v["idx_k"][off[1]:off[1] + n - h])])
    oc, os_ = O.quantise(x, layout)
    assert np.array_equal(scales, os_), np.argwhere(scales != os_)[:5]
    assert np.array_equal(codes, oc), np.argwhere(codes != oc)[:5]
    assert np.array_equal(ik, kx)
    assert v["lengths"].cpu().tolist() == [h, n - h]
    assert cache.length(0) == h and cache.length(1) == n - h
    with pytest.raises(C.Csa2Error) as e:
        C.csa2_append_entries(cache, [1], [1], f32_dev(x[:1]), bf16_dev(kx[:1]))
    assert e.value.status == 3 and cache.length(1) == n - h


@pytest.mark.parametrize("m", [1, 2, 3, 4, 16])
def test_compress_bit_exact(C, m):
    rng = np.random.default_rng(m)
    t = 64 * m
    c = S.f32_to_bf16_bits((rng.standard_normal((t, 512)) * 3).astype(np.float32))
    z = (rng.standard_normal((t, 512)) * rng.choice([0.1, 3, 40], (t, 1))).astype(np.float32)
    z[::5, ::3] += 100.0          # weights that underflow to exactly zero
    z[1::7] = 0.0                 # equal logits
    out = C.csa2_compress(m, bf16_dev(c), f32_dev(z)).cpu().numpy()
    ref = O.compress(c, z, m)
    assert np.array_equal(out.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("m,layout", [(1, 0), (2, 0), (2, 1), (4, 1)])
def test_append_tokens_matches_compress_then_quantise(C, m, layout):
    rng = np.random.default_rng(10 + m)
    n = 333
    c = S.f32_to_bf16_bits(rng.standard_normal((n * m, 512)).astype(np.float32))
    z = rng.standard_normal((n * m, 512)).astype(np.float32)
    kx = S.normal_bf16(S.stream_key(9, S.S_IDXK, 0), 0, n * 128).reshape(n, 128)
    cache = C.Cache(C.config(ratio=m, layout=layout), [n])
    eo = f32_dev(np.zeros((n, 512), np.float32))
    C.csa2_append_tokens(cache, [0], [n * m], bf16_dev(c), f32_dev(z), bf16_dev(kx), eo)
    ent = O.compress(c, z, m)
    assert np.array_equal(eo.cpu().numpy().view(np.uint32), ent.view(np.uint32))
    oc, os_ = O.quantise(ent, layout)
    v = cache.views()
    assert np.array_equal(v["codes"][:n].cpu().numpy(), oc)
    assert np.array_equal(v["scales"][:n].cpu().numpy(), os_)
    with pytest.raises(C.Csa2Error):
        C.csa2_append_tokens(cache, [0], [m + 1 if m > 1 else 1], bf16_dev(c), f32_dev(z),
                             bf16_dev(kx))


def test_device_generator_matches_host():
    import torch
    key = S.stream_key(99, S.S_Q, 3)
    t32 = S.device_fill(torch.empty(12345, dtype=torch.float32, device="cuda"), key, 777)
    tb = S.device_fill(torch.empty(4321, dtype=torch.bfloat16, device="cuda"), key, 5, 8.0)
    assert np.array_equal(t32.cpu().numpy(), S.normal_f32(key, 777, 12345))
    want = S.f32_to_bf16_bits(S.normal_f32(key, 5, 4321) * np.float32(8))
    assert np.array_equal(bf16_host(tb), want)
