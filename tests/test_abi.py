"""The C-ABI library loads and exports every symbol include/csa2.h declares;
host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa2.h")
LIB = os.path.join(ROOT, "fp4_kv_cache_index_gb300", "libcsa2.so")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        import __graft_entry__
        __graft_entry__.build()
    return ctypes.CDLL(LIB)


def declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(csa2_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared()
    assert len(names) >= 18
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    lib.csa2_status_string.restype = ctypes.c_char_p
    assert lib.csa2_status_string(0) == b"ok"
    assert lib.csa2_status_string(3) == b"capacity exceeded"
    assert lib.csa2_status_string(99) == b"unknown status"
    assert lib.csa2_version() == 1


def _cfg(**kw):
    import fp4_kv_cache_index_gb300 as C
    return C.config(**kw)


def test_cache_bytes_and_config_checks(lib):
    import fp4_kv_cache_index_gb300 as C
    f = C.lib.csa2_cache_bytes
    caps = (ctypes.c_int64 * 2)(1000, 24)
    n32 = f(ctypes.byref(_cfg()), 2, caps)
    n16 = f(ctypes.byref(_cfg(layout=1)), 2, caps)
    # 1024 entries: 256 B codes + 16 or 32 B scales + 256 B indexer key each
    assert n32 >= 1024 * (256 + 16 + 256) and n16 - n32 >= 1024 * 16
    assert n16 < 1024 * (256 + 32 + 256) + 64 * 1024
    for bad in (dict(head_dim=256), dict(topk=500), dict(swa=200), dict(ratio=0),
                dict(layout=5), dict(n_heads=48), dict(n_heads=32), dict(idx_heads=16)):
        assert f(ctypes.byref(_cfg(**bad)), 2, caps) == 0
    assert f(ctypes.byref(_cfg()), 0, caps) == 0
    assert f(None, 2, caps) == 0


def test_host_argument_errors(lib):
    import fp4_kv_cache_index_gb300 as C
    L = C.lib
    out = ctypes.c_void_p()
    caps = (ctypes.c_int64 * 1)(16)
    # null / misaligned device memory and bad configs fail before any CUDA call
    assert L.csa2_cache_create(ctypes.byref(_cfg()), 1, caps, None, 1 << 20, None,
                               ctypes.byref(out)) == 1
    assert L.csa2_cache_create(ctypes.byref(_cfg()), 1, caps, ctypes.c_void_p(0x1001), 1 << 20,
                               None, ctypes.byref(out)) == 1
    assert L.csa2_cache_create(ctypes.byref(_cfg(topk=100)), 1, caps, ctypes.c_void_p(0x1000),
                               1 << 20, None, ctypes.byref(out)) == 2
    assert L.csa2_cache_create(ctypes.byref(_cfg()), 1, caps, ctypes.c_void_p(0x1000), 64, None,
                               ctypes.byref(out)) == 3
    assert L.csa2_cache_destroy(None) == 1
    # workspace sizes of an invalid request are 0
    assert L.csa2_index_prefill_workspace_bytes(None, 0, 8) == 0
    assert L.csa2_index_workspace_bytes(None, 8) == 0
    # several readout layers: a null cache or a bad layer count is refused
    # before any launch
    assert L.csa2_sparse_attn_decode_layers(None, 2, 1, None, None, None, None, None, 1.0, None,
                                            None, None, 0, None, None) == 1
    assert L.csa2_sparse_attn_prefill_layers(None, 0, 2, 1, 0, None, None, 0, 0, None, 1.0,
                                             None, None, None, None) == 1
    assert L.csa2_compress(0, 4, 512, None, None, None, None) == 1
    assert L.csa2_compress(2, 0, 512, None, None, None, None) == 0
    assert L.csa2_compress(32, 4, 512, None, None, None, None) == 2
    assert L.csa2_topk(0, None, 0, None, 512, None, None, None, None, 0, None) == 0
    assert L.csa2_topk(1, None, 0, None, 512, None, None, None, None, 0, None) == 1
    nv = (ctypes.c_int64 * 1)(10)
    assert L.csa2_topk(1, ctypes.c_void_p(0x1000), 4, nv, 512, None, ctypes.c_void_p(0x2000),
                       None, None, 0, None) == 1    # n_valid > ld
    assert L.csa2_index_topk_decode(None, 1, None, None, None, None, None, None, 0, None) == 1
    assert L.csa2_sparse_attn_decode(None, 1, None, None, None, None, None, 1.0, None, None,
                                     None, 0, None) == 1
    st = ctypes.c_int32()
    assert L.csa2_get_device_error(None, None, ctypes.byref(st)) == 1
    assert L.csa2_cache_set_wait_limit(None, 100) == 1
    assert L.csa2_cache_inject_fault(None, 0) == 1


def test_every_entry_point_opens_an_nvtx_range():
    """Each C call that can launch or touch the device is wrapped in an NVTX
    range named after it (CSA2_RANGE as its first statement)."""
    src = open(os.path.join(ROOT, "fp4_kv_cache_index_gb300", "csrc", "csa2_api.cu")).read()
    defs = re.findall(r"\ncsa2_status_t (csa2_\w+)\([^)]*\)\s*\{\n(.*)\n", src)
    assert len(defs) >= 25
    for name, first in defs:
        assert first.strip() == "CSA2_RANGE();", name
