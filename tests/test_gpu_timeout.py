"""The timeout path of the bounded waits, exercised without a GPU fault.

With the fault injected (csa2_cache_inject_fault: the indexer's producer
issues no key loads) and a short wait limit, the indexer's MMA and epilogue
waits run out while no copy and no MMA is in flight.  The call must return,
the device error word must read CSA2_ERR_TIMEOUT, and a normal call made
afterwards on the same context must succeed and match the oracle: the
kernel freed its tensor memory and left nothing behind."""
import numpy as np
import pytest

import csa2_synth as S
import oracle as O
from tests._parity import bf16_dev, check_topk, f32_dev

pytestmark = pytest.mark.gpu

TIMEOUT = 6       # CSA2_ERR_TIMEOUT
FAULT_NO_KEY_LOADS = 1


@pytest.mark.parametrize("idx_layout", [0, 1])
def test_wait_runs_out_then_the_context_stays_usable(idx_layout):
    import torch
    import fp4_kv_cache_index_gb300 as C
    lens = [5000, 3000, 777]
    cache = C.Cache(C.config(idx_layout=idx_layout), lens)
    ks = []
    for s, n in enumerate(lens):
        k = S.normal_bf16(S.stream_key(160, S.S_IDXK, s), 0, n * 128).reshape(n, 128)
        e = S.normal_f32(S.stream_key(160, S.S_ENTRIES, s), 0, n * 512).reshape(n, 512)
        C.csa2_append_entries(cache, [s], [n], f32_dev(e), bf16_dev(k))
        ks.append(k)
    qi = S.normal_bf16(S.stream_key(161, S.S_QIDX, 0), 0, 3 * 4096).reshape(3, 32, 128)
    w = S.normal_f32(S.stream_key(161, S.S_W, 0), 0, 3 * 32).reshape(3, 32)
    assert cache.device_error() == 0

    # ---- the injected fault: every wait on the keys runs out (2^20 cycles)
    cache.set_wait_limit(1 << 20)
    cache.inject_fault(FAULT_NO_KEY_LOADS)
    sc = torch.full((3, 5000), 7.0, device="cuda")
    C.csa2_index_scores_decode(cache, bf16_dev(qi), f32_dev(w), sc)
    torch.cuda.synchronize()                  # the kernel ended by itself
    assert cache.device_error() == TIMEOUT
    assert cache.device_error() == 0          # read-and-clear

    # ---- back to normal: the same context computes the right selection
    cache.inject_fault(0)
    cache.set_wait_limit(0)
    idx = C.csa2_index_topk_decode(cache, bf16_dev(qi), f32_dev(w)).cpu().numpy()
    for i, n in enumerate(lens):
        ref = O.index_topk_mxfp4 if idx_layout else O.index_topk
        o_idx, o_sc = ref(ks[i], qi[i], w[i], 512)
        check_topk(idx[i], o_idx, o_sc, 512)
    assert cache.device_error() == 0


def test_wait_limit_and_fault_arguments_are_checked():
    import fp4_kv_cache_index_gb300 as C
    cache = C.Cache(C.config(), [16])
    with pytest.raises(C.Csa2Error):
        cache.set_wait_limit(-1)
    with pytest.raises(C.Csa2Error):
        cache.inject_fault(2)
