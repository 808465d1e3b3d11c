"""Failure detection without a GPU fault (GPU only): a call whose index warp withholds its
items (qsa_debug_stall_next_call) must end on its own once the other roles' bounded waits run
out, report the wait site through the device status word, and leave the context usable."""
import numpy as np
import pytest

import oracle
from helpers import to_device, assert_parity
from top_sparse_attention_row_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SITE_ITEM_FULL = 0x100 | 3          # d=256 kernel: item-record wait
SITE_MLA_ITEM_FULL = 0x100 | 0x23   # MLA kernel: item-record wait


@pytest.fixture(scope="module")
def B():
    from top_sparse_attention_row_gb300 import build, binding
    build.build()
    binding.load_library()
    return binding


def test_stalled_call_times_out_and_the_context_recovers(B):
    import time
    import torch
    w = W.make_tiny()
    q, k, v, idx, tl = to_device(w)
    assert B.device_status() == 0
    B.debug_stall_next_call()
    t0 = time.time()
    B.sparse_prefill(q, k, v, idx, tl, w.scale)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert B.device_status() == SITE_ITEM_FULL
    assert 1.0 < elapsed < 30.0                      # the 2 s wait limit, not a hang
    # the hook is one-shot and the context still works: the next call is exact
    out, lse = B.sparse_prefill(q, k, v, idx, tl, w.scale)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    O, L = oracle.sparse_prefill(w.q, w.k, w.v, w.indices, w.topk_len, w.scale)
    assert_parity(out, lse, O, L, what="after a timed-out call")


def test_stalled_mla_call_times_out(B):
    import torch
    w = W.make_mla(seed=40, n_rows=64, topk=128, n_heads=8, name="mla_stall")
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    q, kv = bf(w.q), bf(w.k.reshape(w.k.shape[0], -1))
    idx = torch.from_numpy(w.indices).cuda()
    B.debug_stall_next_call()
    B.sparse_mla_prefill(q, kv, idx, None, w.scale)
    torch.cuda.synchronize()
    assert B.device_status() == SITE_MLA_ITEM_FULL
    out, lse = B.sparse_mla_prefill(q, kv, idx, None, w.scale)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    O, L = oracle.sparse_mla_prefill(w.q, w.k.reshape(w.k.shape[0], -1), w.indices, None, w.scale)
    assert_parity(out, lse, O, L, what="MLA after a timed-out call")
