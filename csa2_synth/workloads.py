"""The five CSA2 workloads (shapes, seeds, generation recipe) shared by the
benchmark, the parity tests and the oracle runs.  Shapes follow the layer
configuration of the V4.1 report (section 4.2.1: 64 heads of dim 512, 32
indexer heads of dim 128, top-k 512, window 128, ratio 2 in the encoder and
1 in the decoder).  Values are the seeded N(0,1) proxy of this package.

Recipe (per workload, seed = 1234 + workload id):
  * main-KV entries: fp32 [N_b, 512] per sequence b (stream S_ENTRIES, sub b);
    with ``outliers`` the 1% channels chosen by ``choose_channels`` (5 of 512)
    are scaled by 8 in the entries and in the window rows;
  * indexer keys: bf16 [N_b, 128] per sequence (S_IDXK, sub b);
  * indexer queries bf16 [B, 32, 128] and head weights fp32 [B, 32]
    (S_QIDX, S_W);
  * per layer l: queries bf16 [B, 64, 512] (S_Q, sub l) and window rows bf16
    [B, 128, 512] (S_SWA, sub l) for decode, or [T + 127, 512] token rows for
    prefill;
  * ragged lengths (long-context workload): tokens per sequence uniform in
    [512K, 1M] (S_LENGTHS), N_b = tokens // 2.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Tuple

import numpy as np

from . import (S_ENTRIES, S_IDXK, S_Q, S_QIDX, S_SWA, S_W, choose_channels, normal_bf16,
               normal_f32, seq_lengths, stream_key)

HEADS, DIM, IDX_HEADS, IDX_DIM, TOPK, SWA = 64, 512, 32, 128, 512, 128


@dataclass
class Workload:
    wid: int
    name: str
    batch: int
    ctx: int                    # tokens per sequence (decode) or prefix (prefill)
    ratio: int
    layers: int                 # 1 Full + (layers - 1) Reuse
    outliers: bool = False
    ragged: Optional[Tuple[int, int]] = None
    prefill_tokens: int = 0     # new query tokens of a prefill chunk
    notes: str = ""
    _lengths: Optional[np.ndarray] = field(default=None, repr=False)

    @property
    def seed(self) -> int:
        return 1234 + self.wid

    @property
    def prefill(self) -> bool:
        return self.prefill_tokens > 0

    def tokens(self) -> np.ndarray:
        if self._lengths is None:
            if self.ragged:
                self._lengths = seq_lengths(self.seed, self.batch, *self.ragged)
            elif self.prefill:
                self._lengths = np.array([self.ctx + self.prefill_tokens], np.int64)
            else:
                self._lengths = np.full(self.batch, self.ctx, np.int64)
        return self._lengths

    def n_entries(self) -> np.ndarray:
        return self.tokens() // self.ratio

    def n_queries(self) -> int:
        return self.prefill_tokens if self.prefill else self.batch

    def outlier_channels(self) -> np.ndarray:
        return choose_channels(self.seed, DIM, round(0.01 * DIM)) if self.outliers else \
            np.zeros(0, np.int64)

    # ---------------------------------------------------------------- host tensors
    def entries(self, seq: int, first: int = 0, n: Optional[int] = None) -> np.ndarray:
        """fp32 entries [n, 512] of sequence ``seq`` starting at row ``first``."""
        n = int(self.n_entries()[seq]) - first if n is None else n
        x = normal_f32(stream_key(self.seed, S_ENTRIES, seq), first * DIM, n * DIM)
        x = x.reshape(n, DIM)
        ch = self.outlier_channels()
        if len(ch):
            x[:, ch] *= np.float32(8.0)
        return x

    def entry_rows(self, seq: int, rows: np.ndarray) -> np.ndarray:
        """fp32 entries of the given row indices (each generated on its own)."""
        rows = np.asarray(rows, np.int64)
        out = np.empty((len(rows), DIM), np.float32)
        for i, r in enumerate(rows):
            out[i] = self.entries(seq, int(r), 1)[0]
        return out

    def idx_k(self, seq: int, first: int = 0, n: Optional[int] = None) -> np.ndarray:
        n = int(self.n_entries()[seq]) - first if n is None else n
        return normal_bf16(stream_key(self.seed, S_IDXK, seq), first * IDX_DIM,
                           n * IDX_DIM).reshape(n, IDX_DIM)

    def q_idx(self, first: int = 0, n: Optional[int] = None, layer: int = 0) -> np.ndarray:
        """Indexer queries; layer 0 is the Full layer, layer i > 0 the i-th
        Reindex layer (its own indexer query and weights)."""
        n = self.n_queries() - first if n is None else n
        return normal_bf16(stream_key(self.seed, S_QIDX, layer), first * IDX_HEADS * IDX_DIM,
                           n * IDX_HEADS * IDX_DIM).reshape(n, IDX_HEADS, IDX_DIM)

    def w(self, first: int = 0, n: Optional[int] = None, layer: int = 0) -> np.ndarray:
        n = self.n_queries() - first if n is None else n
        return normal_f32(stream_key(self.seed, S_W, layer), first * IDX_HEADS,
                          n * IDX_HEADS).reshape(n, IDX_HEADS)

    def q(self, layer: int, first: int = 0, n: Optional[int] = None) -> np.ndarray:
        n = self.n_queries() - first if n is None else n
        return normal_bf16(stream_key(self.seed, S_Q, layer), first * HEADS * DIM,
                           n * HEADS * DIM).reshape(n, HEADS, DIM)

    def swa_rows_count(self) -> int:
        """Decode: rows per query; prefill: token rows of the chunk's windows."""
        return SWA if not self.prefill else self.prefill_tokens + SWA - 1

    def swa(self, layer: int, first: int = 0, n: Optional[int] = None) -> np.ndarray:
        """Decode: [n, 128, 512] window rows of queries first..; prefill: token
        rows first.. of [T + 127, 512] (row r = position ctx - 127 + r)."""
        if self.prefill:
            n = self.swa_rows_count() - first if n is None else n
            x = normal_f32(stream_key(self.seed, S_SWA, layer), first * DIM, n * DIM)
            x = x.reshape(n, DIM)
        else:
            n = self.batch - first if n is None else n
            x = normal_f32(stream_key(self.seed, S_SWA, layer), first * SWA * DIM,
                           n * SWA * DIM).reshape(n, SWA, DIM)
        ch = self.outlier_channels()
        if len(ch):
            x[..., ch] *= np.float32(8.0)
        from . import f32_to_bf16_bits
        return f32_to_bf16_bits(x)

    @property
    def swa_pos0(self) -> int:
        return self.ctx - (SWA - 1) if self.prefill else 0

    @property
    def pos0(self) -> int:
        return self.ctx if self.prefill else 0


WORKLOADS = {
    0: Workload(0, "decode_b1_ctx4k_m2_full", batch=1, ctx=4096, ratio=2, layers=1),
    1: Workload(1, "decode_b16_ctx32k_m2_full+5reuse", batch=16, ctx=32768, ratio=2, layers=6),
    2: Workload(2, "decode_b64_ctx128k_m1_full+3reuse_outliers", batch=64, ctx=131072, ratio=1,
                layers=4, outliers=True),
    3: Workload(3, "decode_b4_ctx1m_m2_ragged_full", batch=4, ctx=1048576, ratio=2, layers=1,
                ragged=(524288, 1048576)),
    4: Workload(4, "prefill_8k_on_128k_m2_full+3reuse", batch=1, ctx=131072, ratio=2, layers=4,
                prefill_tokens=8192),
}


# ---------------------------------------------------------------- device tensors
def _dev(shape, dtype):
    import torch
    return torch.empty(*shape, dtype=dtype, device="cuda")


def _outlier_scale(wl: Workload, t):
    ch = wl.outlier_channels()
    if len(ch):
        import torch
        idx = torch.as_tensor(ch, device=t.device)
        t[..., idx] *= 8
    return t


def dev_entries(wl: Workload, seq: int, first: int, n: int):
    import torch
    from . import device_fill
    t = device_fill(_dev((n, DIM), torch.float32), stream_key(wl.seed, S_ENTRIES, seq),
                    first * DIM)
    return _outlier_scale(wl, t)


def dev_idx_k(wl: Workload, seq: int, first: int, n: int):
    import torch
    from . import device_fill
    return device_fill(_dev((n, IDX_DIM), torch.bfloat16), stream_key(wl.seed, S_IDXK, seq),
                       first * IDX_DIM)


def dev_q_idx(wl: Workload, first: int = 0, n: Optional[int] = None, layer: int = 0):
    import torch
    from . import device_fill
    n = wl.n_queries() - first if n is None else n
    return device_fill(_dev((n, IDX_HEADS, IDX_DIM), torch.bfloat16),
                       stream_key(wl.seed, S_QIDX, layer), first * IDX_HEADS * IDX_DIM)


def dev_w(wl: Workload, first: int = 0, n: Optional[int] = None, layer: int = 0):
    import torch
    from . import device_fill
    n = wl.n_queries() - first if n is None else n
    return device_fill(_dev((n, IDX_HEADS), torch.float32), stream_key(wl.seed, S_W, layer),
                       first * IDX_HEADS)


def dev_q(wl: Workload, layer: int, first: int = 0, n: Optional[int] = None):
    import torch
    from . import device_fill
    n = wl.n_queries() - first if n is None else n
    return device_fill(_dev((n, HEADS, DIM), torch.bfloat16), stream_key(wl.seed, S_Q, layer),
                       first * HEADS * DIM)


def dev_swa(wl: Workload, layer: int):
    import torch
    from . import device_fill
    shape = (wl.swa_rows_count(), DIM) if wl.prefill else (wl.batch, SWA, DIM)
    t = device_fill(_dev(shape, torch.bfloat16), stream_key(wl.seed, S_SWA, layer), 0)
    return _outlier_scale(wl, t)


def fill_cache(wl: Workload, cache, chunk_rows: int = 1 << 16):
    """Appends every sequence's entries and indexer keys through
    csa2_append_entries, ``chunk_rows`` rows at a time."""
    from fp4_kv_cache_index_gb300 import csa2_append_entries
    for seq, n in enumerate(wl.n_entries()):
        for r0 in range(0, int(n), chunk_rows):
            m = min(chunk_rows, int(n) - r0)
            csa2_append_entries(cache, [seq], [m], dev_entries(wl, seq, r0, m),
                                dev_idx_k(wl, seq, r0, m))
