"""CPU oracle of the CSA2 attention step over an FP4 global KV cache.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs may import this package.  The
product path (``fp4_kv_cache_index_gb300``) never does.

The arithmetic lives in ``csa2_oracle.c`` (plain C, OpenMP, fp64 where the
method is real-valued, fp32 where a float decides an integer).  This module
builds it with gcc, binds it with ctypes and composes the per-query steps
(index -> top-k -> attention, Full / Reuse layers, causal prefill) in the
order the pages describe them:

* Full mode computes the index scores and a fresh top-k; Reuse mode takes the
  latest top-k of its group unchanged and only runs attention
  ("DeepSeek-V4.1-Flash" report, section 2.3.1).
* Every layer uses its own query and its own sliding-window KV (same section).
* A query at absolute position p sees compressed entry s iff the block of s is
  complete, (s + 1) * m - 1 <= p, and the window rows [max(s0, p - W + 1), p]
  (report section 3.2.2, SWA Bounded Replay; s0 = 0 without replay).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa2_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libcsa2_oracle.so")
_lock = threading.Lock()
_lib = None

LAYOUT_L32_UE8M0 = 0
LAYOUT_L16_E4M3 = 1


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, OpenMP, no fp contraction)."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                               os.path.getmtime(_SRC[:-1] + "h"))):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i64, i32, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_float
            sig = {
                "orc_num_threads": ([], i32),
                "orc_e2m1_value": ([i32], f32),
                "orc_e2m1_encode": ([f32], i32),
                "orc_e4m3_value": ([i32], f32),
                "orc_e4m3_encode": ([f32], i32),
                "orc_ue8m0_value": ([i32], f32),
                "orc_ue8m0_for_amax": ([f32], i32),
                "orc_group": ([i32], i32),
                "orc_quantise": ([i64, i32, i32, P, P, P], None),
                "orc_dequantise": ([i64, i32, i32, P, P, P], None),
                "orc_entry_bytes": ([i32, i32], ctypes.c_double),
                "orc_bytes_per_token": ([i32, P, P], ctypes.c_double),
                "orc_expf": ([f32], f32),
                "orc_compress": ([i64, i32, i32, P, P, P], None),
                "orc_index_scores": ([i64, i32, i32, P, P, P, P], None),
                "orc_topk": ([i64, P, i32, P], i32),
                "orc_bf16_round": ([f32], f32),
                "orc_ue8m0_for_amax_e4m3": ([f32], i32),
                "orc_swa_fp8_quantise": ([i64, P, P, P, P], None),
                "orc_swa_fp8_dequantise": ([i64, P, P, P, P], None),
                "orc_bf16_round_n": ([i64, P, P], None),
                "orc_sparse_attention": ([i32, i32, i32, P, P, P, i64, i32, P, i32, P,
                                          f32, P, P, P], None),
            }
            for name, (args, res) in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def _p(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def num_threads() -> int:
    return int(lib().orc_num_threads())


# ---------------------------------------------------------------- codec
def e2m1_value(code: int) -> float:
    return float(lib().orc_e2m1_value(int(code)))


def e2m1_encode(v: float) -> int:
    return int(lib().orc_e2m1_encode(float(v)))


def e4m3_value(b: int) -> float:
    return float(lib().orc_e4m3_value(int(b)))


def e4m3_encode(v: float) -> int:
    return int(lib().orc_e4m3_encode(float(v)))


def ue8m0_value(b: int) -> float:
    return float(lib().orc_ue8m0_value(int(b)))


def ue8m0_for_amax(a: float) -> int:
    return int(lib().orc_ue8m0_for_amax(float(a)))


def group(layout: int) -> int:
    return int(lib().orc_group(int(layout)))


def quantise(x: np.ndarray, layout: int):
    """fp32 [n, dim] -> (codes uint8 [n, dim/2], scales uint8 [n, dim/g])."""
    x = _c(x, np.float32)
    n, dim = x.shape
    g = group(layout)
    codes = np.zeros((n, dim // 2), np.uint8)
    scales = np.zeros((n, dim // g), np.uint8)
    lib().orc_quantise(n, dim, layout, _p(x), _p(codes), _p(scales))
    return codes, scales


def dequantise(codes: np.ndarray, scales: np.ndarray, layout: int) -> np.ndarray:
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    n = codes.shape[0]
    dim = codes.shape[1] * 2
    out = np.zeros((n, dim), np.float32)
    lib().orc_dequantise(n, dim, layout, _p(codes), _p(scales), _p(out))
    return out


def swa_fp8_quantise(rows_bf16):
    """bf16 window rows [n, 512] -> FP8 rows: E4M3 codes [n, 448], bf16 RoPE
    channels [n, 64], UE8M0 scales [n, 8] (one per 64 channels, byte 7
    unused).  See orc_swa_fp8_quantise for the reading of the format."""
    x = _c(rows_bf16, np.uint16).reshape(-1, 512)
    n = x.shape[0]
    codes = np.zeros((n, 448), np.uint8)
    rope = np.zeros((n, 64), np.uint16)
    scales = np.zeros((n, 8), np.uint8)
    lib().orc_swa_fp8_quantise(n, _p(x), _p(codes), _p(rope), _p(scales))
    return codes, rope, scales


def swa_fp8_dequantise(codes, rope, scales) -> np.ndarray:
    codes = _c(codes, np.uint8)
    rope = _c(rope, np.uint16)
    scales = _c(scales, np.uint8)
    n = codes.shape[0]
    out = np.zeros((n, 512), np.float32)
    lib().orc_swa_fp8_dequantise(n, _p(codes), _p(rope), _p(scales), _p(out))
    return out


def swa_fp8_round_bf16(rows_bf16) -> np.ndarray:
    """Window rows through FP8 and back, as bf16 bits (every dequantised
    value is a bf16 value): what the attention reads from an FP8 window."""
    d = swa_fp8_dequantise(*swa_fp8_quantise(rows_bf16))
    shape = np.shape(rows_bf16)
    return (d.view(np.uint32) >> 16).astype(np.uint16).reshape(shape)


def entry_bytes(dim: int, layout: int) -> float:
    return float(lib().orc_entry_bytes(dim, layout))


def bytes_per_token(ratios, bytes_per_entry) -> float:
    r = _c(ratios, np.int32)
    b = _c(bytes_per_entry, np.float64)
    return float(lib().orc_bytes_per_token(len(r), _p(r), _p(b)))


# ---------------------------------------------------------------- compressor
def expf(x: float) -> float:
    return float(lib().orc_expf(float(x)))


def compress(c_bf16: np.ndarray, z: np.ndarray, m: int) -> np.ndarray:
    """Tokens [n*m, dim] (bf16 bits, fp32 logits) -> entries fp32 [n, dim]."""
    c_bf16 = _c(c_bf16, np.uint16)
    z = _c(z, np.float32)
    t, dim = c_bf16.shape
    n = t // m
    out = np.zeros((n, dim), np.float32)
    lib().orc_compress(n, m, dim, _p(c_bf16), _p(z), _p(out))
    return out


# ---------------------------------------------------------------- indexer
def index_scores(k_bf16: np.ndarray, q_bf16: np.ndarray, w: np.ndarray) -> np.ndarray:
    """fp64 scores of one query (q [heads, d]) against keys k [n, d]."""
    k_bf16 = _c(k_bf16, np.uint16)
    q_bf16 = _c(q_bf16, np.uint16)
    w = _c(w, np.float32)
    n, d = k_bf16.shape
    heads = q_bf16.shape[0]
    out = np.zeros(n, np.float64)
    lib().orc_index_scores(n, heads, d, _p(k_bf16), _p(q_bf16), _p(w), _p(out))
    return out


def topk(scores_f32: np.ndarray, k: int) -> np.ndarray:
    """Top-k of fp32 scores: ties to the lower index, ascending, -1 padded."""
    s = _c(scores_f32, np.float32)
    out = np.zeros(k, np.int32)
    lib().orc_topk(len(s), _p(s), k, _p(out))
    return out


def bf16_round(x) -> np.ndarray:
    """fp32 -> nearest bf16 value (ties to even), returned as fp32."""
    a = _c(np.atleast_1d(x), np.float32)
    out = np.zeros_like(a)
    lib().orc_bf16_round_n(a.size, _p(a), _p(out))
    return out.reshape(np.shape(x))


# ---------------------------------------------------------------- attention
def sparse_attention(q_bf16, codes, scales, layout, idx, swa_bf16, scale):
    """One query: q [heads, dim] over the selected entries (idx, -1 skipped)
    and the window rows swa [n_swa, dim].  Returns (out bf16 bits [heads, dim],
    out fp64 [heads, dim], lse fp64 [heads])."""
    q_bf16 = _c(q_bf16, np.uint16)
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    idx = _c(idx, np.int32)
    heads, dim = q_bf16.shape
    swa = _c(swa_bf16, np.uint16).reshape(-1, dim) if swa_bf16 is not None else \
        np.zeros((0, dim), np.uint16)
    out_b = np.zeros((heads, dim), np.uint16)
    out_d = np.zeros((heads, dim), np.float64)
    lse = np.zeros(heads, np.float64)
    lib().orc_sparse_attention(heads, dim, layout, _p(q_bf16), _p(codes), _p(scales),
                               codes.shape[0], len(idx), _p(idx), swa.shape[0], _p(swa),
                               float(scale), _p(out_b), _p(out_d), _p(lse))
    return out_b, out_d, lse


def attention_epilogue(out_d, lse, sink=None, rope_pos=None, rope_base: float = 10000.0,
                       rope_dims: int = 64):
    """Epilogue variants of the readout ("DeepSeek-V4" blog reading, section
    4.3), applied in fp64 to one query's core attention output:

    * attention sink: a per-head learnable logit z'_h whose exp joins the
      softmax denominator, s_j = exp(l_j) / (sum_k exp(l_k) + exp(z'_h)), so a
      head's weights may sum to less than 1 (the sink carries no value);
    * output RoPE(-i): the last `rope_dims` channels of the output, taken as
      interleaved pairs (2t, 2t+1) with frequency base^(-2t / rope_dims), are
      rotated by the angle of position -i, so the output carries relative
      rather than absolute position.

    out_d: fp64 [heads, dim] and lse: fp64 [heads] from sparse_attention
    (natural log of the denominator without the sink).  Returns
    (out bf16 bits, out fp64, lse fp64 of the full denominator)."""
    out = np.array(out_d, np.float64, copy=True)
    lse = np.asarray(lse, np.float64)
    if sink is not None:
        z = np.asarray(sink, np.float64)
        lse_all = np.logaddexp(lse, z)
        # a head with neither candidates nor sink keeps its empty softmax:
        # output 0, lse -inf (as without a sink)
        empty = np.isneginf(lse_all)
        factor = np.exp(lse - np.where(empty, 0.0, lse_all))
        out *= np.where(empty, 0.0, factor)[:, None]
        lse = lse_all
    if rope_pos is not None:
        d0 = out.shape[1] - rope_dims
        t = np.arange(rope_dims // 2, dtype=np.float64)
        phi = -float(rope_pos) * rope_base ** (-2.0 * t / rope_dims)
        c, s_ = np.cos(phi), np.sin(phi)
        a = out[:, d0::2].copy()
        b = out[:, d0 + 1::2].copy()
        out[:, d0::2] = a * c - b * s_
        out[:, d0 + 1::2] = a * s_ + b * c
    rounded = bf16_round(out.astype(np.float32))
    bits = (rounded.view(np.uint32) >> 16).astype(np.uint16)
    return bits, out, lse


# ---------------------------------------------------------------- composition
def visible_entries(n_ent: int, m: int, pos=None) -> int:
    """Entries a query sees: all of them in decode (the query is the newest
    token); in prefill, entry s is visible at position p iff (s+1)*m-1 <= p."""
    if pos is None:
        return int(n_ent)
    return int(min(n_ent, (int(pos) + 1) // m))


def index_topk(k_bf16, q_bf16, w, k, n_vis=None):
    """Full-layer selection for one query: fp64 scores over the visible
    entries, rounded to fp32 (the precision the selection is made in), then
    the top-k.  Returns (idx [k], scores fp64 [n_vis])."""
    n_vis = k_bf16.shape[0] if n_vis is None else n_vis
    sc = index_scores(k_bf16[:n_vis], q_bf16, w)
    return topk(sc.astype(np.float32), k), sc


def mxfp4_round_bf16(x_bf16) -> np.ndarray:
    """Rows of 128 bf16 channels onto the OCP MXFP4 grid ("DeepSeek-V4.1-
    Flash" report, section 2.4.4: FP4 indexer queries and keys; one UE8M0
    scale per 32 channels, the L32 rule of `quantise`), returned as bf16
    bits (every E2M1 code times a power-of-two scale is a bf16 value)."""
    x = np.asarray(x_bf16, np.uint16)
    shape = x.shape
    f = (x.astype(np.uint32) << 16).view(np.float32).reshape(-1, shape[-1])
    codes, scales = quantise(f, LAYOUT_L32_UE8M0)
    d = dequantise(codes, scales, LAYOUT_L32_UE8M0)
    return (d.view(np.uint32) >> 16).astype(np.uint16).reshape(shape)


def index_topk_mxfp4(k_bf16, q_bf16, w, k, n_vis=None):
    """Full-layer selection with MXFP4 indexer keys and queries: the keys and
    every query head rounded to the MXFP4 grid, then the fp64 score of the
    dequantised values, rounded to fp32 for the top-k.  Returns (idx [k],
    fp64 scores [n_vis])."""
    n_vis = k_bf16.shape[0] if n_vis is None else n_vis
    kq = mxfp4_round_bf16(np.asarray(k_bf16)[:n_vis])
    qq = mxfp4_round_bf16(q_bf16)
    sc = index_scores(kq, qq, w)
    return topk(sc.astype(np.float32), k), sc


def index_topk_bf16(k_bf16, q_bf16, w, k, n_vis=None):
    """Selection on bf16-rounded scores ("DeepSeek-V4" blog reading, section
    7): fp64 scores -> fp32 -> bf16, then the top-k with ties (now frequent)
    to the lower index.  Returns (idx [k], bf16 scores as fp32 [n_vis],
    fp64 scores [n_vis])."""
    n_vis = k_bf16.shape[0] if n_vis is None else n_vis
    sc = index_scores(k_bf16[:n_vis], q_bf16, w)
    b = bf16_round(sc.astype(np.float32))
    return topk(b, k), b, sc


def recall(selected, reference) -> float:
    """Fraction of the reference selection (valid indices) that `selected`
    also holds."""
    r = np.asarray(reference)
    r = r[r >= 0]
    if len(r) == 0:
        return 1.0
    s = np.asarray(selected)
    return float(np.isin(r, s[s >= 0]).sum()) / len(r)


def swa_rows(pos: int, window: int, row0_pos: int = 0):
    """Window rows of a query at absolute position ``pos`` as absolute
    positions [max(row0_pos, pos - window + 1), pos] (report section 3.2.2)."""
    lo = max(row0_pos, pos - window + 1)
    return lo, pos + 1


# ---------------------------------------------------------------- hierarchical sparse indexer
def hsi_pool(scores_f32, n_vis: int, block: int = 8, max_blocks: int = 2048) -> np.ndarray:
    """Candidate pool of the Hierarchical Sparse Indexer ("DeepSeek-V4.1-Flash"
    report, section 2.3.2): each block of `block` consecutive positions gets
    the maximum index score among its visible positions; the `max_blocks`
    blocks with the highest block scores are kept (ties to the lower block
    index, the same selection rule as the entries' top-k).  Returns the kept
    block indices in ascending order, padded with -1 to `max_blocks`."""
    s = np.asarray(scores_f32, np.float32)[:n_vis]
    n_blocks = (n_vis + block - 1) // block
    bmax = np.full(n_blocks, -np.inf, np.float32)
    for b in range(n_blocks):
        bmax[b] = s[b * block:(b + 1) * block].max()
    return topk(bmax, max_blocks)


def pool_positions(pool_blocks, n_vis: int, block: int = 8) -> np.ndarray:
    """Visible positions covered by the pool blocks, ascending."""
    b = np.asarray(pool_blocks)
    b = b[b >= 0]
    pos = (b[:, None] * block + np.arange(block)[None, :]).ravel()
    return pos[pos < n_vis]


def reindex_topk(k_bf16, q_bf16, w, pool_blocks, n_vis: int, k: int = 512, block: int = 8):
    """Reindex mode (same section): the layer's own indexer query scores only
    the pool positions (fp64, rounded to fp32 for the decision) and keeps the
    top-k of them, ties to the lower position, ascending, -1 padded.
    Returns (idx [k], fp64 scores of the pool positions, the positions)."""
    pos = pool_positions(pool_blocks, n_vis, block)
    sc = index_scores(np.asarray(k_bf16)[pos], q_bf16, w)
    sel = topk(sc.astype(np.float32), k)
    out = np.full(k, -1, np.int32)
    n = int((sel >= 0).sum())
    out[:n] = pos[sel[:n]]
    return out, sc, pos
