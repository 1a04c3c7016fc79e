"""GB300-native CSA2 sparse attention over an FP4 global KV cache.

Thin Python binding of ``libcsa2.so`` (the C ABI in ``include/csa2.h``).  It
only marshals arguments: torch tensors become device pointers, the current
torch stream becomes the launch stream, and output tensors are created with
torch when the caller passes none.  Every step of the attention path runs in
the library's CUDA kernels; there is no fallback.  If the library has not been
built the import of this module raises.

Function names follow the C ABI (``csa2_index_topk_decode`` ...).  ``Cache``
owns the device buffer of one CSA2 group's global cache and its handle.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# CSA2_DEBUG=1 loads the bounds-checked build (libcsa2_debug.so, built by
# _build.build(debug=True)); otherwise the normal one.
LIB_PATH = os.path.join(_HERE, "libcsa2_debug.so" if os.environ.get("CSA2_DEBUG") == "1"
                        else "libcsa2.so")

CSA2_KV_L32_UE8M0 = 0
CSA2_KV_L16_E4M3 = 1

STATUS = {0: "CSA2_OK", 1: "CSA2_ERR_INVALID_ARG", 2: "CSA2_ERR_UNSUPPORTED",
          3: "CSA2_ERR_CAPACITY", 4: "CSA2_ERR_CUDA", 5: "CSA2_ERR_OOM",
          6: "CSA2_ERR_TIMEOUT", 7: "CSA2_ERR_DEVICE"}


class Csa2Error(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [("n_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("idx_heads", ctypes.c_int32), ("idx_dim", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("swa", ctypes.c_int32),
                ("ratio", ctypes.c_int32), ("layout", ctypes.c_int32),
                ("idx_layout", ctypes.c_int32)]


def config(n_heads=64, head_dim=512, idx_heads=32, idx_dim=128, topk=512, swa=128, ratio=1,
           layout=CSA2_KV_L32_UE8M0, idx_layout=0) -> Config:
    """Layer shapes of the V4.1 report, section 4.2.1, as defaults;
    idx_layout 1 keeps the indexer keys in MXFP4 (CSA2_IDX_MXFP4)."""
    return Config(n_heads, head_dim, idx_heads, idx_dim, topk, swa, ratio, layout, idx_layout)


class AttnOpts(ctypes.Structure):
    """csa2_attn_opts_t: attention sink and output RoPE(-i)."""
    _fields_ = [("sink", ctypes.c_void_p), ("rope_pos", ctypes.c_void_p),
                ("rope_out", ctypes.c_int32), ("rope_base", ctypes.c_double),
                ("swa_codes", ctypes.c_void_p), ("swa_rope", ctypes.c_void_p),
                ("swa_scales", ctypes.c_void_p)]


class CacheViews(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("idx_k", ctypes.c_void_p), ("lengths", ctypes.c_void_p),
                ("entry_offset", ctypes.POINTER(ctypes.c_int64)), ("total", ctypes.c_int64),
                ("batch", ctypes.c_int32), ("group", ctypes.c_int32),
                ("idx_codes", ctypes.c_void_p), ("idx_scales", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                          "(the CSA2 path has no CPU fallback)")
    L = ctypes.CDLL(LIB_PATH)
    P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    pcfg = ctypes.POINTER(Config)
    sigs = {
        "csa2_version": ([], i32),
        "csa2_status_string": ([i32], ctypes.c_char_p),
        "csa2_cache_bytes": ([pcfg, i32, P], sz),
        "csa2_cache_create": ([pcfg, i32, P, P, sz, P, ctypes.POINTER(P)], i32),
        "csa2_cache_destroy": ([P], i32),
        "csa2_cache_set_index_sms": ([P, i32], i32),
        "csa2_cache_set_wait_limit": ([P, i64], i32),
        "csa2_cache_inject_fault": ([P, i32], i32),
        "csa2_cache_reset": ([P, P], i32),
        "csa2_cache_length": ([P, i32, ctypes.POINTER(i64)], i32),
        "csa2_cache_views": ([P, ctypes.POINTER(CacheViews)], i32),
        "csa2_compress": ([i32, i64, i32, P, P, P, P], i32),
        "csa2_append_entries": ([P, i32, P, P, P, P, P], i32),
        "csa2_append_tokens": ([P, i32, P, P, P, P, P, P, P], i32),
        "csa2_index_workspace_bytes": ([P, i32], sz),
        "csa2_index_scores_decode": ([P, i32, P, P, P, P, i64, P, P], i32),
        "csa2_index_topk_decode": ([P, i32, P, P, P, P, P, P, sz, P], i32),
        "csa2_index_topk_prefill": ([P, i32, i32, i64, P, P, P, P, P, sz, P], i32),
        "csa2_index_topk_decode_static": ([P, i32, P, P, P, P, P, P], i32),
        "csa2_index_topk": ([P, i32, P, P, P, P, P, P, P, sz, P], i32),
        "csa2_index_scores_prefill": ([P, i32, i32, i64, P, P, P, i64, P, P], i32),
        "csa2_index_prefill_workspace_bytes": ([P, i32, i32], sz),
        "csa2_index_scores_decode_bf16": ([P, i32, P, P, P, P, i64, P, P], i32),
        "csa2_topk_bf16": ([i32, P, i64, P, i32, P, P, P, P, sz, P], i32),
        "csa2_index_topk_decode_bf16": ([P, i32, P, P, P, P, P, P, sz, P], i32),
        "csa2_sparse_attn_decode_ex": ([P, i32, P, P, P, P, P, ctypes.c_float, P, P, P, sz, P,
                                        P], i32),
        "csa2_sparse_attn_decode_layers": ([P, i32, i32, P, P, P, P, P, ctypes.c_float, P, P, P, sz,
                                            P, P], i32),
        "csa2_sparse_attn_prefill_ex": ([P, i32, i32, i64, P, P, i64, i64, P, ctypes.c_float, P,
                                         P, P, P], i32),
        "csa2_sparse_attn_prefill_layers": ([P, i32, i32, i32, i64, P, P, i64, i64, P,
                                             ctypes.c_float, P, P, P, P], i32),
        "csa2_swa_fp8_quantise": ([i64, P, P, P, P, P], i32),
        "csa2_hsi_pool_workspace_bytes": ([i32, i64], sz),
        "csa2_hsi_pool": ([i32, P, i64, P, i32, i32, P, P, sz, P], i32),
        "csa2_index_reindex_workspace_bytes": ([P, i32, i32], sz),
        "csa2_index_topk_reindex_decode": ([P, i32, P, P, P, P, i32, P, P, P, sz, P], i32),
        "csa2_topk_workspace_bytes": ([i32, i64], sz),
        "csa2_topk": ([i32, P, i64, P, i32, P, P, P, P, sz, P], i32),
        "csa2_sparse_attn_workspace_bytes": ([P, i32], sz),
        "csa2_sparse_attn_decode": ([P, i32, P, P, P, P, P, ctypes.c_float, P, P, P, sz, P], i32),
        "csa2_sparse_attn_prefill": ([P, i32, i32, i64, P, P, i64, i64, P, ctypes.c_float, P, P,
                                      P], i32),
        "csa2_get_device_error": ([P, P, ctypes.POINTER(i32)], i32),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    return L


lib = _load()


def _check(st: int, what: str):
    if st != 0:
        raise Csa2Error(st, what)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _i32_array(xs: Optional[Sequence[int]]):
    if xs is None:
        return None
    return (ctypes.c_int32 * len(xs))(*[int(x) for x in xs])


def _i64_array(xs: Sequence[int]):
    return (ctypes.c_int64 * len(xs))(*[int(x) for x in xs])


class Cache:
    """One CSA2 group's global KV cache in a torch-owned device buffer."""

    def __init__(self, cfg: Config, capacity: Sequence[int], device=None, stream=None):
        self.cfg = cfg
        self.batch = len(capacity)
        caps = _i64_array(capacity)
        nbytes = lib.csa2_cache_bytes(ctypes.byref(cfg), self.batch, caps)
        if nbytes == 0:
            raise Csa2Error(1, "csa2_cache_bytes")
        device = torch.device("cuda") if device is None else torch.device(device)
        self.buffer = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
        self._off = (-self.buffer.data_ptr()) % 256
        self.handle = ctypes.c_void_p()
        _check(lib.csa2_cache_create(ctypes.byref(cfg), self.batch, caps,
                                     ctypes.c_void_p(self.buffer.data_ptr() + self._off),
                                     nbytes, _stream(stream), ctypes.byref(self.handle)),
               "csa2_cache_create")

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value:
            lib.csa2_cache_destroy(h)
            self.handle = None

    def length(self, seq: int) -> int:
        n = ctypes.c_int64()
        _check(lib.csa2_cache_length(self.handle, seq, ctypes.byref(n)), "csa2_cache_length")
        return n.value

    def reset(self, stream=None):
        _check(lib.csa2_cache_reset(self.handle, _stream(stream)), "csa2_cache_reset")

    def set_index_sms(self, n_sms: int):
        """At most n_sms SMs for the indexer's grid (0: all); see
        csa2_cache_set_index_sms."""
        _check(lib.csa2_cache_set_index_sms(self.handle, n_sms), "csa2_cache_set_index_sms")

    def set_wait_limit(self, cycles: int):
        """Bounded-wait limit of this cache's kernels in SM cycles (0: the
        default); see csa2_cache_set_wait_limit."""
        _check(lib.csa2_cache_set_wait_limit(self.handle, cycles), "csa2_cache_set_wait_limit")

    def inject_fault(self, fault: int):
        """0: none; 1: the indexers issue no key loads (tests of the timeout
        path); see csa2_cache_inject_fault."""
        _check(lib.csa2_cache_inject_fault(self.handle, fault), "csa2_cache_inject_fault")

    def views(self) -> dict:
        """codes [total, 256] u8, scales [total, 512/g] u8, idx_k [total, 128]
        bf16, lengths [batch] int32, entry_offset (list), group."""
        v = CacheViews()
        _check(lib.csa2_cache_views(self.handle, ctypes.byref(v)), "csa2_cache_views")
        base = self.buffer.data_ptr()
        total = v.total

        def sl(ptr, nbytes):
            o = ptr - base
            return self.buffer[o:o + nbytes]

        g = v.group
        mx = bool(v.idx_codes)
        return {
            "codes": sl(v.codes, total * 256).view(total, 256),
            "scales": sl(v.scales, total * (512 // g)).view(total, 512 // g),
            "idx_k": None if mx else sl(v.idx_k, total * 256).view(torch.bfloat16).view(total, 128),
            "idx_codes": sl(v.idx_codes, total * 64).view(total, 64) if mx else None,
            "idx_scales": sl(v.idx_scales, total * 4).view(total, 4) if mx else None,
            "lengths": sl(v.lengths, 4 * self.batch).view(torch.int32),
            "entry_offset": [v.entry_offset[i] for i in range(self.batch + 1)],
            "group": g,
        }

    def device_error(self, stream=None) -> int:
        st = ctypes.c_int32()
        _check(lib.csa2_get_device_error(self.handle, _stream(stream), ctypes.byref(st)),
               "csa2_get_device_error")
        return st.value


# ------------------------------------------------------------------ compress / append
def csa2_compress(ratio: int, c_tok: torch.Tensor, z_tok: torch.Tensor,
                  out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    t, dim = c_tok.shape
    n_out = t // ratio
    if out is None:
        out = torch.empty(n_out, dim, dtype=torch.float32, device=c_tok.device)
    _check(lib.csa2_compress(ratio, n_out, dim, _ptr(c_tok), _ptr(z_tok), _ptr(out),
                             _stream(stream)), "csa2_compress")
    return out


def csa2_append_entries(cache: Cache, seq_ids: Sequence[int], n_new: Sequence[int],
                        entries: torch.Tensor, idx_k: torch.Tensor, stream=None):
    _check(lib.csa2_append_entries(cache.handle, len(seq_ids), _i32_array(seq_ids),
                                   _i32_array(n_new), _ptr(entries), _ptr(idx_k),
                                   _stream(stream)), "csa2_append_entries")


def csa2_append_tokens(cache: Cache, seq_ids: Sequence[int], n_tok: Sequence[int],
                       c_tok: torch.Tensor, z_tok: torch.Tensor, idx_k: torch.Tensor,
                       entries_out: Optional[torch.Tensor] = None, stream=None):
    _check(lib.csa2_append_tokens(cache.handle, len(seq_ids), _i32_array(seq_ids),
                                  _i32_array(n_tok), _ptr(c_tok), _ptr(z_tok), _ptr(idx_k),
                                  _ptr(entries_out), _stream(stream)), "csa2_append_tokens")


# ------------------------------------------------------------------ indexer + top-k
def csa2_index_workspace_bytes(cache: Cache, n_queries: int) -> int:
    return int(lib.csa2_index_workspace_bytes(cache.handle, n_queries))


def _workspace(nbytes: int, device, workspace):
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)
    return workspace


def csa2_index_scores_decode(cache: Cache, q_idx: torch.Tensor, w: torch.Tensor,
                             scores: torch.Tensor, seq_ids: Optional[Sequence[int]] = None,
                             key_hist: Optional[torch.Tensor] = None,
                             stream=None) -> torch.Tensor:
    """scores: fp32 [n_queries, ld] (ld a multiple of 4, >= every length);
    key_hist: optional int32 [n_queries, 2048] score-key histogram output."""
    _check(lib.csa2_index_scores_decode(cache.handle, q_idx.shape[0], _ptr(q_idx), _ptr(w),
                                        _i32_array(seq_ids), _ptr(scores), scores.shape[1],
                                        _ptr(key_hist), _stream(stream)),
           "csa2_index_scores_decode")
    return scores


def csa2_index_topk_decode(cache: Cache, q_idx: torch.Tensor, w: torch.Tensor,
                           seq_ids: Optional[Sequence[int]] = None,
                           topk_idx: Optional[torch.Tensor] = None,
                           topk_score: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    nq = q_idx.shape[0]
    dev = q_idx.device
    if topk_idx is None:
        topk_idx = torch.empty(nq, cache.cfg.topk, dtype=torch.int32, device=dev)
    ws = _workspace(csa2_index_workspace_bytes(cache, nq), dev, workspace)
    _check(lib.csa2_index_topk_decode(cache.handle, nq, _ptr(q_idx), _ptr(w),
                                      _i32_array(seq_ids), _ptr(topk_idx), _ptr(topk_score),
                                      _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "csa2_index_topk_decode")
    return topk_idx


def csa2_index_topk(cache: Cache, q_idx: torch.Tensor, w: torch.Tensor,
                    seq_of_q: Optional[Sequence[int]], q_pos: Sequence[int],
                    topk_idx: Optional[torch.Tensor] = None,
                    topk_score: Optional[torch.Tensor] = None,
                    workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Selection for queries at token positions q_pos of sequences seq_of_q
    (host lists; seq_of_q None: query i reads sequence i)."""
    nq = q_idx.shape[0]
    dev = q_idx.device
    if topk_idx is None:
        topk_idx = torch.empty(nq, cache.cfg.topk, dtype=torch.int32, device=dev)
    ws = _workspace(csa2_index_workspace_bytes(cache, nq), dev, workspace)
    _check(lib.csa2_index_topk(cache.handle, nq, _ptr(q_idx), _ptr(w), _i32_array(seq_of_q),
                               _i64_array(q_pos), _ptr(topk_idx), _ptr(topk_score), _ptr(ws),
                               ws.numel() * ws.element_size(), _stream(stream)),
           "csa2_index_topk")
    return topk_idx


def csa2_index_scores_prefill(cache: Cache, seq: int, pos0: int, q_idx: torch.Tensor,
                              w: torch.Tensor, scores: torch.Tensor,
                              key_hist: Optional[torch.Tensor] = None, stream=None):
    """scores: fp32 [n_queries, ld] (ld a multiple of 4, >= the length);
    key_hist: int32 [n_queries, 2048] score-key histograms (bf16 keys)."""
    _check(lib.csa2_index_scores_prefill(cache.handle, seq, q_idx.shape[0], pos0, _ptr(q_idx),
                                         _ptr(w), _ptr(scores), scores.shape[1], _ptr(key_hist),
                                         _stream(stream)), "csa2_index_scores_prefill")
    return scores


def csa2_index_prefill_workspace_bytes(cache: Cache, seq: int, n_queries: int) -> int:
    return int(lib.csa2_index_prefill_workspace_bytes(cache.handle, seq, n_queries))


def csa2_index_topk_prefill(cache: Cache, seq: int, pos0: int, q_idx: torch.Tensor,
                            w: torch.Tensor, topk_idx: Optional[torch.Tensor] = None,
                            topk_score: Optional[torch.Tensor] = None,
                            workspace: Optional[torch.Tensor] = None,
                            stream=None) -> torch.Tensor:
    nq = q_idx.shape[0]
    dev = q_idx.device
    if topk_idx is None:
        topk_idx = torch.empty(nq, cache.cfg.topk, dtype=torch.int32, device=dev)
    ws = _workspace(csa2_index_prefill_workspace_bytes(cache, seq, nq), dev, workspace)
    _check(lib.csa2_index_topk_prefill(cache.handle, seq, nq, pos0, _ptr(q_idx), _ptr(w),
                                       _ptr(topk_idx), _ptr(topk_score), _ptr(ws),
                                       ws.numel() * ws.element_size(), _stream(stream)),
           "csa2_index_topk_prefill")
    return topk_idx


def csa2_topk_workspace_bytes(n_rows: int, max_valid: int) -> int:
    return int(lib.csa2_topk_workspace_bytes(n_rows, max_valid))


def csa2_topk(scores: torch.Tensor, n_valid: Sequence[int], k: int,
              idx_out: Optional[torch.Tensor] = None, score_out: Optional[torch.Tensor] = None,
              key_hist: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
              stream=None):
    rows, ld = scores.shape
    if idx_out is None:
        idx_out = torch.empty(rows, k, dtype=torch.int32, device=scores.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.csa2_topk(rows, _ptr(scores), ld, _i64_array(n_valid), k, _ptr(key_hist),
                         _ptr(idx_out), _ptr(score_out), _ptr(workspace), ws_bytes,
                         _stream(stream)), "csa2_topk")
    return idx_out


# ------------------------------------------------------------------ attention
def csa2_sparse_attn_workspace_bytes(cache: Cache, n_queries: int) -> int:
    return int(lib.csa2_sparse_attn_workspace_bytes(cache.handle, n_queries))


def csa2_sparse_attn_decode(cache: Cache, q: torch.Tensor, swa_kv: Optional[torch.Tensor],
                            topk_idx: torch.Tensor, scale: float,
                            swa_len: Optional[torch.Tensor] = None,
                            seq_ids: Optional[Sequence[int]] = None,
                            out: Optional[torch.Tensor] = None,
                            lse: Optional[torch.Tensor] = None,
                            workspace: Optional[torch.Tensor] = None,
                            sink: Optional[torch.Tensor] = None,
                            rope_pos: Optional[torch.Tensor] = None, rope_base: float = 0.0,
                            swa_fp8=None, stream=None) -> torch.Tensor:
    """workspace=None allocates one of csa2_sparse_attn_workspace_bytes; pass
    an empty tensor to run without (one CTA per query).  sink: fp32 [n_heads]
    per-head sink logits; rope_pos: int64 [n_queries] positions i for the
    output RoPE(-i)."""
    nq = q.shape[0]
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = torch.empty(max(16, csa2_sparse_attn_workspace_bytes(cache, nq)),
                                dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    args = (cache.handle, nq, _i32_array(seq_ids), _ptr(q), _ptr(swa_kv), _ptr(swa_len),
            _ptr(topk_idx), float(scale), _ptr(out), _ptr(lse),
            _ptr(workspace) if ws_bytes else None, ws_bytes)
    if sink is None and rope_pos is None and swa_fp8 is None:
        _check(lib.csa2_sparse_attn_decode(*args, _stream(stream)), "csa2_sparse_attn_decode")
    else:
        f8 = swa_fp8 if swa_fp8 is not None else (None, None, None)
        opts = AttnOpts(_ptr(sink), _ptr(rope_pos), 1 if rope_pos is not None else 0,
                        float(rope_base), _ptr(f8[0]), _ptr(f8[1]), _ptr(f8[2]))
        _check(lib.csa2_sparse_attn_decode_ex(*args, ctypes.byref(opts), _stream(stream)),
               "csa2_sparse_attn_decode_ex")
    return out


def csa2_sparse_attn_decode_layers(cache: Cache, qs: Sequence[torch.Tensor],
                                   swa_kvs: Optional[Sequence[Optional[torch.Tensor]]],
                                   topk_idx: torch.Tensor, scale: float,
                                   outs: Sequence[torch.Tensor],
                                   lses: Optional[Sequence[Optional[torch.Tensor]]] = None,
                                   swa_len: Optional[torch.Tensor] = None,
                                   seq_ids: Optional[Sequence[int]] = None,
                                   workspace: Optional[torch.Tensor] = None,
                                   sinks: Optional[Sequence[Optional[torch.Tensor]]] = None,
                                   rope_pos: Optional[torch.Tensor] = None, rope_base: float = 0.0,
                                   swa_fp8s=None, stream=None):
    """The readout of several layers of a group in one launch (per layer:
    queries, window rows or their FP8 form, sink, outputs); workspace as for
    csa2_sparse_attn_decode."""
    L = len(qs)
    nq = qs[0].shape[0]
    if workspace is None:
        workspace = torch.empty(max(16, csa2_sparse_attn_workspace_bytes(cache, nq)),
                                dtype=torch.uint8, device=qs[0].device)
    ws_bytes = workspace.numel() * workspace.element_size()
    arr = lambda xs: (ctypes.c_void_p * L)(*[_ptr(x) for x in xs])
    swa_arr = arr(swa_kvs) if swa_kvs is not None else None
    lse_arr = arr(lses) if lses is not None else None
    keep = []
    opts_arr = None
    if sinks is not None or rope_pos is not None or swa_fp8s is not None:
        ptrs = []
        for l in range(L):
            f8 = swa_fp8s[l] if swa_fp8s is not None and swa_fp8s[l] is not None else (None, None, None)
            o = AttnOpts(_ptr(sinks[l] if sinks is not None else None), _ptr(rope_pos),
                         1 if rope_pos is not None else 0, float(rope_base),
                         _ptr(f8[0]), _ptr(f8[1]), _ptr(f8[2]))
            keep.append(o)
            ptrs.append(ctypes.cast(ctypes.pointer(o), ctypes.c_void_p))
        opts_arr = (ctypes.c_void_p * L)(*ptrs)
    _check(lib.csa2_sparse_attn_decode_layers(cache.handle, L, nq, _i32_array(seq_ids), arr(qs),
                                              swa_arr, _ptr(swa_len), _ptr(topk_idx),
                                              float(scale), arr(outs), lse_arr,
                                              _ptr(workspace) if ws_bytes else None, ws_bytes,
                                              opts_arr, _stream(stream)),
           "csa2_sparse_attn_decode_layers")
    return outs


def csa2_sparse_attn_prefill(cache: Cache, seq: int, pos0: int, q: torch.Tensor,
                             swa_kv: Optional[torch.Tensor], swa_pos0: int,
                             topk_idx: torch.Tensor, scale: float,
                             out: Optional[torch.Tensor] = None,
                             lse: Optional[torch.Tensor] = None,
                             sink: Optional[torch.Tensor] = None, rope_out: bool = False,
                             rope_base: float = 0.0, swa_fp8=None, stream=None) -> torch.Tensor:
    """rope_out: rotate the last 64 output channels by RoPE(-(pos0 + i));
    swa_fp8: (codes, rope, scales) of csa2_swa_fp8_quantise instead of
    swa_kv."""
    nq = q.shape[0]
    if out is None:
        out = torch.empty_like(q)
    n_rows = swa_fp8[0].shape[0] if swa_fp8 is not None else (
        swa_kv.shape[0] if swa_kv is not None else 0)
    args = (cache.handle, seq, nq, pos0, _ptr(q), _ptr(swa_kv), swa_pos0, n_rows,
            _ptr(topk_idx), float(scale), _ptr(out), _ptr(lse))
    if sink is None and not rope_out and swa_fp8 is None:
        _check(lib.csa2_sparse_attn_prefill(*args, _stream(stream)), "csa2_sparse_attn_prefill")
    else:
        f8 = swa_fp8 if swa_fp8 is not None else (None, None, None)
        opts = AttnOpts(_ptr(sink), None, 1 if rope_out else 0, float(rope_base),
                        _ptr(f8[0]), _ptr(f8[1]), _ptr(f8[2]))
        _check(lib.csa2_sparse_attn_prefill_ex(*args, ctypes.byref(opts), _stream(stream)),
               "csa2_sparse_attn_prefill_ex")
    return out


def csa2_sparse_attn_prefill_layers(cache: Cache, seq: int, pos0: int,
                                    qs: Sequence[torch.Tensor],
                                    swa_kvs: Optional[Sequence[Optional[torch.Tensor]]],
                                    swa_pos0: int, topk_idx: torch.Tensor, scale: float,
                                    outs: Sequence[torch.Tensor],
                                    lses: Optional[Sequence[Optional[torch.Tensor]]] = None,
                                    sinks: Optional[Sequence[Optional[torch.Tensor]]] = None,
                                    rope_out: bool = False, rope_base: float = 0.0,
                                    swa_fp8s=None, stream=None):
    """The prefill readout of several layers of a group in one launch (per
    layer: queries, window rows or their FP8 form, sink, outputs)."""
    L = len(qs)
    nq = qs[0].shape[0]
    n_rows = 0
    for l in range(L):
        if swa_fp8s is not None and swa_fp8s[l] is not None:
            n_rows = swa_fp8s[l][0].shape[0]
        elif swa_kvs is not None and swa_kvs[l] is not None:
            n_rows = swa_kvs[l].shape[0]
    arr = lambda xs: (ctypes.c_void_p * L)(*[_ptr(x) for x in xs])
    swa_arr = arr(swa_kvs) if swa_kvs is not None else None
    lse_arr = arr(lses) if lses is not None else None
    keep = []
    opts_arr = None
    if sinks is not None or rope_out or swa_fp8s is not None:
        ptrs = []
        for l in range(L):
            f8 = swa_fp8s[l] if swa_fp8s is not None and swa_fp8s[l] is not None else (None, None, None)
            o = AttnOpts(_ptr(sinks[l] if sinks is not None else None), None,
                         1 if rope_out else 0, float(rope_base),
                         _ptr(f8[0]), _ptr(f8[1]), _ptr(f8[2]))
            keep.append(o)
            ptrs.append(ctypes.cast(ctypes.pointer(o), ctypes.c_void_p))
        opts_arr = (ctypes.c_void_p * L)(*ptrs)
    _check(lib.csa2_sparse_attn_prefill_layers(cache.handle, seq, L, nq, pos0, arr(qs), swa_arr,
                                               swa_pos0, n_rows, _ptr(topk_idx), float(scale),
                                               arr(outs), lse_arr, opts_arr, _stream(stream)),
           "csa2_sparse_attn_prefill_layers")
    return outs


# ------------------------------------------------------------------ hierarchical sparse indexer
def csa2_hsi_pool(scores: torch.Tensor, n_valid: Sequence[int], max_blocks: int = 2048,
                  block: int = 8, pool_blocks: Optional[torch.Tensor] = None,
                  workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """scores: fp32 [rows, ld] of a Full layer; returns int32 [rows, max_blocks]
    kept block indices (ascending, -1 padded)."""
    rows, ld = scores.shape
    if pool_blocks is None:
        pool_blocks = torch.empty(rows, max_blocks, dtype=torch.int32, device=scores.device)
    workspace = _workspace(int(lib.csa2_hsi_pool_workspace_bytes(rows, max(n_valid, default=0))),
                           scores.device, workspace)
    _check(lib.csa2_hsi_pool(rows, _ptr(scores), ld, _i64_array(n_valid), block, max_blocks,
                             _ptr(pool_blocks), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream(stream)),
           "csa2_hsi_pool")
    return pool_blocks


def csa2_index_topk_reindex_decode(cache: Cache, q_idx: torch.Tensor, w: torch.Tensor,
                                   pool_blocks: torch.Tensor,
                                   seq_ids: Optional[Sequence[int]] = None,
                                   topk_idx: Optional[torch.Tensor] = None,
                                   topk_score: Optional[torch.Tensor] = None,
                                   workspace: Optional[torch.Tensor] = None,
                                   stream=None) -> torch.Tensor:
    """Reindex-layer top-k inside each query's pool (pool_blocks from
    csa2_hsi_pool, one row per query); returns int32 [n_queries, topk]."""
    nq, max_blocks = pool_blocks.shape
    if topk_idx is None:
        topk_idx = torch.empty(nq, cache.cfg.topk, dtype=torch.int32, device=q_idx.device)
    workspace = _workspace(int(lib.csa2_index_reindex_workspace_bytes(cache.handle, nq, max_blocks)),
                           q_idx.device, workspace)
    _check(lib.csa2_index_topk_reindex_decode(cache.handle, nq, _ptr(q_idx), _ptr(w),
                                              _i32_array(seq_ids), _ptr(pool_blocks), max_blocks,
                                              _ptr(topk_idx), _ptr(topk_score), _ptr(workspace),
                                              workspace.numel() * workspace.element_size(),
                                              _stream(stream)),
           "csa2_index_topk_reindex_decode")
    return topk_idx


# ------------------------------------------------------------------ bf16-rounded scores
def csa2_index_scores_decode_bf16(cache: Cache, q_idx: torch.Tensor, w: torch.Tensor,
                                  scores: torch.Tensor, seq_ids: Optional[Sequence[int]] = None,
                                  key_hist: Optional[torch.Tensor] = None,
                                  stream=None) -> torch.Tensor:
    """scores: bf16 (or int16) [n_queries, ld], ld a multiple of 8."""
    _check(lib.csa2_index_scores_decode_bf16(cache.handle, q_idx.shape[0], _ptr(q_idx), _ptr(w),
                                             _i32_array(seq_ids), _ptr(scores), scores.shape[1],
                                             _ptr(key_hist), _stream(stream)),
           "csa2_index_scores_decode_bf16")
    return scores


def csa2_topk_bf16(scores: torch.Tensor, n_valid: Sequence[int], k: int,
                   idx_out: Optional[torch.Tensor] = None,
                   score_out: Optional[torch.Tensor] = None,
                   key_hist: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    rows, ld = scores.shape
    if idx_out is None:
        idx_out = torch.empty(rows, k, dtype=torch.int32, device=scores.device)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.csa2_topk_bf16(rows, _ptr(scores), ld, _i64_array(n_valid), k, _ptr(key_hist),
                              _ptr(idx_out), _ptr(score_out), _ptr(workspace), nbytes,
                              _stream(stream)),
           "csa2_topk_bf16")
    return idx_out


def csa2_index_topk_decode_bf16(cache: Cache, q_idx: torch.Tensor, w: torch.Tensor,
                                seq_ids: Optional[Sequence[int]] = None,
                                topk_idx: Optional[torch.Tensor] = None,
                                topk_score: Optional[torch.Tensor] = None,
                                workspace: Optional[torch.Tensor] = None,
                                stream=None) -> torch.Tensor:
    nq = q_idx.shape[0]
    dev = q_idx.device
    if topk_idx is None:
        topk_idx = torch.empty(nq, cache.cfg.topk, dtype=torch.int32, device=dev)
    ws = _workspace(csa2_index_workspace_bytes(cache, nq), dev, workspace)
    _check(lib.csa2_index_topk_decode_bf16(cache.handle, nq, _ptr(q_idx), _ptr(w),
                                           _i32_array(seq_ids), _ptr(topk_idx), _ptr(topk_score),
                                           _ptr(ws), ws.numel() * ws.element_size(),
                                           _stream(stream)),
           "csa2_index_topk_decode_bf16")
    return topk_idx


# ------------------------------------------------------------------ FP8 window rows
def csa2_swa_fp8_quantise(rows: torch.Tensor, stream=None):
    """bf16 rows [..., 512] -> (codes u8 [n, 448], rope bf16 [n, 64],
    scales u8 [n, 8]) with n the number of rows."""
    r = rows.reshape(-1, 512)
    n = r.shape[0]
    codes = torch.empty(n, 448, dtype=torch.uint8, device=rows.device)
    rope = torch.empty(n, 64, dtype=torch.bfloat16, device=rows.device)
    scales = torch.empty(n, 8, dtype=torch.uint8, device=rows.device)
    _check(lib.csa2_swa_fp8_quantise(n, _ptr(r), _ptr(codes), _ptr(rope), _ptr(scales),
                                     _stream(stream)), "csa2_swa_fp8_quantise")
    return codes, rope, scales
