"""Seeded synthetic inputs for the CSA2 decode / prefill workloads.

This module is the one piece that the CUDA path's harness and the CPU oracle
both use.  It holds no arithmetic of the attention method itself: it only
turns (seed, stream, sub-stream, element index) into numbers.

Generator
---------
* SplitMix64 (Steele, Lea and Flood, "Fast Splittable Pseudorandom Number
  Generators", OOPSLA 2014), used in its counter-based form: draw ``d`` of a
  stream with key ``K`` is ``mix64(K + (d + 1) * GAMMA)``.
* Normal proxy: the Irwin-Hall sum of twelve uniforms (the classic
  "sum twelve uniforms, subtract six" method).  Each value takes three draws,
  each draw gives four 16-bit uniforms, and
  ``z = (sum_of_twelve_u16 - 393210) / 65536``, which has mean 0 and
  variance ``1 - 2**-32``.  Every step is integer arithmetic followed by one
  exact scaling, so the host (numpy) and device (``gen.cu``) twins produce
  identical bits.  ``z`` is exact in fp32; bf16 tensors take it rounded to
  nearest-even.

Stream ids name the tensors of one workload; ``sub`` selects the sequence or
layer.  Element ``i`` of a tensor is the flat row-major index.
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_GAMMA2 = np.uint64(0xD1B54A32D192ED03)
IH_MEAN = 393210          # 12 * 32767.5
IH_SCALE = 2.0 ** -16

# stream ids (one per tensor kind of a workload)
S_ENTRIES = 1      # fp32 compressed main-KV entries, sub = sequence
S_IDXK = 2         # bf16 indexer keys, sub = sequence
S_QIDX = 3         # bf16 indexer queries, sub = 0
S_W = 4            # fp32 indexer head weights, sub = 0
S_Q = 5            # bf16 attention queries, sub = layer
S_SWA = 6          # bf16 sliding-window KV rows, sub = layer
S_TOKC = 7         # bf16 uncompressed token KV (compressor input), sub = sequence
S_TOKZ = 8         # fp32 compressor logits, sub = sequence
S_LENGTHS = 9      # integer sequence lengths
S_OUTLIER = 10     # outlier channel choice
S_SCORES = 11      # fp32 scores for stand-alone top-k cases


def _mix64(z):
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int, sub: int = 0) -> int:
    """64-bit key of one tensor stream (same formula as the device twin)."""
    with np.errstate(over="ignore"):
        k0 = _mix64(np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + GAMMA)
        k1 = _mix64(k0 ^ (np.uint64(stream) * _GAMMA2))
        k = _mix64(k1 + np.uint64(sub) * GAMMA)
    return int(k)


def draws(key: int, first: int, n: int) -> np.ndarray:
    """Raw 64-bit draws ``first .. first+n-1`` of the stream with ``key``."""
    d = np.arange(first + 1, first + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(np.uint64(key) + d * GAMMA)


def _u16_sum(r: np.ndarray) -> np.ndarray:
    m = np.uint64(0xFFFF)
    return ((r & m) + ((r >> np.uint64(16)) & m) + ((r >> np.uint64(32)) & m)
            + (r >> np.uint64(48))).astype(np.int64)


def normal_f32(key: int, first: int, n: int, chunk: int = 1 << 22) -> np.ndarray:
    """Elements ``first .. first+n-1`` of an fp32 N(0,1)-proxy tensor."""
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, chunk):
        c = min(chunk, n - s)
        r = draws(key, 3 * (first + s), 3 * c).reshape(c, 3)
        tot = _u16_sum(r[:, 0]) + _u16_sum(r[:, 1]) + _u16_sum(r[:, 2])
        out[s:s + c] = (tot - IH_MEAN).astype(np.float32) * np.float32(IH_SCALE)
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest-even) and return the 16-bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bias = ((b >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((b + bias) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(key: int, first: int, n: int) -> np.ndarray:
    """bf16 bit patterns of the N(0,1)-proxy tensor (fp32 value rounded RNE)."""
    return f32_to_bf16_bits(normal_f32(key, first, n))


def uniform_int(key: int, first: int, n: int, lo: int, hi: int) -> np.ndarray:
    """Integers in [lo, hi] (inclusive), one draw each (modulo reduction)."""
    span = np.uint64(hi - lo + 1)
    return (draws(key, first, n) % span).astype(np.int64) + lo


def choose_channels(seed: int, n_channels: int, count: int) -> np.ndarray:
    """``count`` distinct channel indices out of ``n_channels`` (partial
    Fisher-Yates over the outlier stream), returned sorted."""
    key = stream_key(seed, S_OUTLIER, 0)
    perm = np.arange(n_channels, dtype=np.int64)
    r = draws(key, 0, count)
    for i in range(count):
        j = i + int(r[i] % np.uint64(n_channels - i))
        perm[i], perm[j] = perm[j], perm[i]
    return np.sort(perm[:count])


def seq_lengths(seed: int, batch: int, lo: int, hi: int) -> np.ndarray:
    """Per-sequence token counts drawn uniformly in [lo, hi]."""
    return uniform_int(stream_key(seed, S_LENGTHS, 0), 0, batch, lo, hi)


# ---------------------------------------------------------------- device twin
_dev_lib = None


def _device_lib():
    global _dev_lib
    if _dev_lib is None:
        import ctypes
        import os
        path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libcsa2synth.so")
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(path)
        for name in ("csa2_synth_fill_f32", "csa2_synth_fill_bf16"):
            fn = getattr(L, name)
            fn.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_float,
                           ctypes.c_void_p, ctypes.c_void_p]
            fn.restype = ctypes.c_int
        _dev_lib = L
    return _dev_lib


def device_fill(t, key: int, first: int = 0, scale: float = 1.0, stream=None):
    """Fill a contiguous CUDA tensor (float32 or bfloat16) with elements
    ``first ..`` of the stream with ``key``; ``scale`` must be a power of two.
    Bit-identical to ``normal_f32`` / ``normal_bf16`` times ``scale``."""
    import ctypes
    import torch
    assert t.is_cuda and t.is_contiguous()
    s = stream if stream is not None else torch.cuda.current_stream()
    L = _device_lib()
    fn = L.csa2_synth_fill_f32 if t.dtype == torch.float32 else L.csa2_synth_fill_bf16
    assert t.dtype in (torch.float32, torch.bfloat16)
    rc = fn(key & 0xFFFFFFFFFFFFFFFF, first, t.numel(), scale, ctypes.c_void_p(t.data_ptr()),
            ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise RuntimeError(f"csa2_synth fill failed: cuda error {rc}")
    return t
