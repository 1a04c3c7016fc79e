"""GPU top-k (csa2_topk) against the oracle's full sort on identical fp32
scores: the index lists must be identical (ties to the lower index,
ascending order, -1 padding)."""
import numpy as np
import pytest

import oracle as O
from tests._parity import f32_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def C():
    import fp4_kv_cache_index_gb300 as C
    return C


def _rows(kind, n, rng):
    if kind == "normal":
        return rng.standard_normal(n).astype(np.float32)
    if kind == "ints":          # many exact ties everywhere
        return rng.integers(-30, 30, n).astype(np.float32)
    if kind == "equal":         # one crowded bin, all ties
        return np.full(n, 2.5, np.float32)
    if kind == "crowded":       # > 8192 keys share the top 11 bits, distinct below
        return (1.0 + rng.random(n) * 2.0 ** -3).astype(np.float32)
    if kind == "signed_zero":
        x = rng.choice(np.float32([0.0, -0.0, 1.0, -1.0]), n)
        return x.astype(np.float32)
    if kind == "relu_like":     # many exact zeros, as after ReLU with few heads
        x = rng.standard_normal(n).astype(np.float32)
        x[x < 1.0] = 0.0
        return x
    raise ValueError(kind)


@pytest.mark.parametrize("kind", ["normal", "ints", "equal", "crowded", "signed_zero", "relu_like"])
@pytest.mark.parametrize("n", [0, 1, 511, 512, 513, 4097, 70001])
def test_topk_matches_full_sort(C, kind, n):
    rng = np.random.default_rng(n + len(kind))
    s = _rows(kind, max(n, 1), rng)[:n]
    ld = max(4, (n + 3) // 4 * 4)
    buf = np.zeros((1, ld), np.float32)
    buf[0, :n] = s
    sc = f32_dev(buf)
    import torch
    so = torch.zeros(1, 512, dtype=torch.float32, device="cuda")
    got = C.csa2_topk(sc, [n], 512, score_out=so).cpu().numpy()[0]
    want = O.topk(s, 512)
    assert np.array_equal(got, want)
    keff = min(n, 512)
    assert np.array_equal(so.cpu().numpy()[0, :keff], s[got[:keff]])


@pytest.mark.parametrize("k", [128, 512, 2048])
def test_ragged_rows_odd_stride(C, k):
    rng = np.random.default_rng(k)
    ns = [0, 5, k - 1, k, k + 1, 3000, 9999, 262147]
    ld = 262147 + 2            # odd row stride: rows are not 16-byte aligned
    buf = rng.standard_normal((len(ns), ld)).astype(np.float32)
    buf[2, :] = np.round(buf[2, :] * 4)
    got = C.csa2_topk(f32_dev(buf), ns, k).cpu().numpy()
    for r, n in enumerate(ns):
        assert np.array_equal(got[r], O.topk(buf[r, :n], k)), r


def test_long_row(C):
    rng = np.random.default_rng(3)
    n = 524288
    s = (rng.standard_normal(n) * 50).astype(np.float32)
    got = C.csa2_topk(f32_dev(s[None]), [n], 512).cpu().numpy()[0]
    assert np.array_equal(got, O.topk(s, 512))


@pytest.mark.parametrize("kind", ["normal", "ints", "equal", "crowded", "relu_like"])
def test_topk_with_key_histogram(C, kind):
    """Given the score-key histogram, the selection is the same."""
    import torch
    from tests.test_gpu_index import _key_hist
    rng = np.random.default_rng(7)
    n = 131072
    s = _rows(kind, n, rng)
    kh = torch.from_numpy(_key_hist(s).astype(np.int32)[None]).cuda()
    got = C.csa2_topk(f32_dev(s[None]), [n], 512, key_hist=kh).cpu().numpy()[0]
    assert np.array_equal(got, O.topk(s, 512))
    ws = torch.empty(C.csa2_topk_workspace_bytes(1, n), dtype=torch.uint8, device="cuda")
    got = C.csa2_topk(f32_dev(s[None]), [n], 512, key_hist=kh, workspace=ws).cpu().numpy()[0]
    assert np.array_equal(got, O.topk(s, 512))


def test_segmented_ragged_rows(C):
    """Segmented candidate search over rows of different lengths (some shorter
    than one segment, some not a multiple of it) and a crowded row."""
    import torch
    from tests.test_gpu_index import _key_hist
    rng = np.random.default_rng(11)
    ns = [100, 512, 513, 16383, 16385, 70001, 140000, 140000]
    ld = 140000
    buf = rng.standard_normal((len(ns), ld)).astype(np.float32)
    buf[7] = np.round(buf[7])               # crowded: falls back to the row scan
    kh = np.stack([_key_hist(buf[r, :n]) for r, n in enumerate(ns)]).astype(np.int32)
    ws = torch.empty(C.csa2_topk_workspace_bytes(len(ns), max(ns)), dtype=torch.uint8,
                     device="cuda")
    got = C.csa2_topk(f32_dev(buf), ns, 512, key_hist=torch.from_numpy(kh).cuda(),
                      workspace=ws).cpu().numpy()
    for r, n in enumerate(ns):
        assert np.array_equal(got[r], O.topk(buf[r, :n], 512)), r


def test_segmented_unaligned_rows(C):
    """Segmented candidate search over rows that are not 16-byte aligned (odd
    row stride), where the segment kernel stages the scores with plain loads
    instead of asynchronous 16-byte copies."""
    import torch
    from tests.test_gpu_index import _key_hist
    rng = np.random.default_rng(12)
    ns = [513, 9000, 16385, 70001]
    ld = 70001 + 2
    buf = rng.standard_normal((len(ns), ld)).astype(np.float32)
    kh = np.stack([_key_hist(buf[r, :n]) for r, n in enumerate(ns)]).astype(np.int32)
    ws = torch.empty(C.csa2_topk_workspace_bytes(len(ns), max(ns)), dtype=torch.uint8,
                     device="cuda")
    got = C.csa2_topk(f32_dev(buf), ns, 512, key_hist=torch.from_numpy(kh).cuda(),
                      workspace=ws).cpu().numpy()
    for r, n in enumerate(ns):
        assert np.array_equal(got[r], O.topk(buf[r, :n], 512)), r


@pytest.mark.parametrize("mode", ["plain", "key_hist", "segments"])
def test_many_rows_two_per_sm(C, mode):
    """A launch of 512 rows or more runs 512 threads a row, two rows per SM:
    rows of every kind and length (empty, below, at and above k, crowded,
    ties, signed zeros), with the row kernel's own histogram, with the
    score-key histogram, and with segments read back."""
    import torch
    from tests.test_gpu_index import _key_hist
    rng = np.random.default_rng(23)
    kinds = ["normal", "ints", "equal", "crowded", "signed_zero", "relu_like"]
    lens = [0, 5, 511, 512, 513, 3000, 8193, 20000]
    R, ld = 640, 20004
    buf = np.zeros((R, ld), np.float32)
    ns = []
    for r in range(R):
        n = lens[r % len(lens)]
        buf[r, :n] = _rows(kinds[(r // len(lens)) % len(kinds)], max(n, 1), rng)[:n]
        ns.append(n)
    kh = ws = None
    if mode != "plain":
        kh = torch.from_numpy(np.stack([_key_hist(buf[r, :n]) for r, n in enumerate(ns)])
                              .astype(np.int32)).cuda()
    if mode == "segments":
        ws = torch.empty(C.csa2_topk_workspace_bytes(R, max(ns)), dtype=torch.uint8,
                         device="cuda")
    got = C.csa2_topk(f32_dev(buf), ns, 512, key_hist=kh, workspace=ws).cpu().numpy()
    for r, n in enumerate(ns):
        assert np.array_equal(got[r], O.topk(buf[r, :n], 512)), r
