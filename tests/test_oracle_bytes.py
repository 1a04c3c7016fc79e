"""Closed-form pins: the 890 bytes/token global KV and its ~1/4 ratio to
V4-Flash ("DeepSeek-V4.1-Flash" report, abstract and Figure 1(b); layer
layout in section 4.2.1; neshdevtech article section 3.1 for the V4-Flash
entry sizes), and the compression / candidate-set arithmetic."""
import itertools

import pytest

import oracle as O
from tests._golden import numbers

G = numbers()
L32, L16 = O.LAYOUT_L32_UE8M0, O.LAYOUT_L16_E4M3


def _v41_bytes(main_layout, idx_layout):
    main = O.entry_bytes(G["kv_latent_dim"], main_layout)
    idx = O.entry_bytes(G["indexer_head_dim"], idx_layout)
    ratios = [G["encoder_ratio"]] * G["encoder_full_layers"] + \
             [G["decoder_ratio"]] * G["decoder_full_layers"]
    return O.bytes_per_token(ratios, [main + idx] * len(ratios))


def test_entry_sizes():
    assert O.entry_bytes(512, L16) == 288       # E2M1 + E4M3 per 16
    assert O.entry_bytes(512, L32) == 272       # E2M1 + UE8M0 per 32
    assert O.entry_bytes(128, L32) == 68        # MXFP4 indexer key


def test_890_bytes_per_token_pins_the_layout():
    assert _v41_bytes(L16, L32) == G["global_kv_bytes_per_token"]
    others = {(a, b): _v41_bytes(a, b) for a, b in itertools.product((L32, L16), repeat=2)}
    hits = [k for k, v in others.items() if v == G["global_kv_bytes_per_token"]]
    assert hits == [(L16, L32)]      # only E4M3/16 main KV + MXFP4 indexer K gives 890
    assert sorted(others.values()) == [850.0, 860.0, 890.0, 900.0]


def test_v4flash_ratio_is_about_four():
    v4_idx = O.entry_bytes(G["indexer_head_dim"], L32)
    ratios = [G["v4_csa_ratio"]] * G["v4_csa_layers"] + [G["v4_hca_ratio"]] * G["v4_hca_layers"]
    bpe = [G["v4_main_entry_bytes"] + v4_idx] * G["v4_csa_layers"] + \
          [G["v4_main_entry_bytes"]] * G["v4_hca_layers"]
    v4 = O.bytes_per_token(ratios, bpe)
    assert v4 == pytest.approx(3514.25)
    assert round(v4 / G["global_kv_bytes_per_token"]) == G["v4flash_over_v41_kv_ratio"]


def test_v4_main_entry_is_584():
    # 448 non-RoPE channels in FP8, 64 RoPE channels in BF16, 8 FP8 scale bytes
    assert 448 * 1 + 64 * 2 + 8 == G["v4_main_entry_bytes"]


def test_compression_and_pool_arithmetic():
    assert O.visible_entries(4096 // 2, 2) == 2048
    assert 32768 // 2 == 16384 and 1048576 // 2 == 524288
    assert G["hsi_blocks"] * G["hsi_block_positions"] == G["hsi_pool"]
    assert G["swa_window"] + G["attention_topk"] == G["candidate_set"]
    # causal visibility: at position p only complete blocks are visible
    assert [O.visible_entries(10, 2, p) for p in range(6)] == [0, 1, 1, 2, 2, 3]
    assert O.visible_entries(10, 2, 1000) == 10
    assert [O.visible_entries(10, 1, p) for p in range(3)] == [1, 2, 3]


def test_kv_latent_bound_fits_the_format():
    assert abs(G["kv_latent_dim"] ** 0.5 - G["kv_latent_abs_bound"]) < 0.05
    assert G["kv_latent_abs_bound"] < G["fp4_max_magnitude"]


@pytest.mark.parametrize("window", [1, 4, 128])
@pytest.mark.parametrize("row0", [0, 3, 150])
def test_window_rows_by_enumeration(window, row0):
    """The window rows of a query at position p: the last `window` tokens up
    to and including p, none before the replay start ("DeepSeek-V4.1-Flash"
    report, section 3.2.2, bounded replay), checked against enumerating the
    positions one by one."""
    for p in range(row0, row0 + 400):
        lo, hi = O.swa_rows(p, window, row0)
        want = [j for j in range(0, p + 1) if j > p - window and j >= row0]
        assert list(range(lo, hi)) == want, (p, window, row0)
    # the window of the 128K workload: 128 rows (the query's own token last)
    assert O.swa_rows(131071, G["swa_window"]) == (131071 - 127, 131072)
