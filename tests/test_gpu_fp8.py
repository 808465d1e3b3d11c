"""qsa_sparse_prefill_fp8 (e4m3 K/V with a scale per page and KV head, dequantised in the gather)
against the FP8 oracle (GPU only).  Bounds: O max-abs 2e-2, LSE relative 1e-3 (helpers.py)."""
import numpy as np
import pytest

import oracle
from helpers import to_device, assert_parity
from top_sparse_attention_row_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from top_sparse_attention_row_gb300 import build, binding
    build.build()
    binding.load_library()
    return binding


def run(B, w, union_g=0, n_kv_slots=0):
    import torch
    q, _, _, idx, tl = to_device(w)
    m = w.meta
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out, lse = B.sparse_prefill_fp8(q, t(m["k8"]), t(m["v8"]), t(m["k_scale"]), t(m["v_scale"]),
                                    m["fp8_page_size"], idx, tl, w.scale, union_g=union_g,
                                    n_kv_slots=n_kv_slots)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    return out, lse


def ref(w, rows=None, n_kv_slots=0):
    m = w.meta
    rows = np.arange(w.n_rows) if rows is None else rows
    return oracle.sparse_prefill_fp8_rows(w.q, m["k8"], m["v8"], m["k_scale"], m["v_scale"],
                                          m["fp8_page_size"], w.indices, w.topk_len, w.scale, rows,
                                          n_kv_slots)


def test_fp8_tiny(B):
    w = W.with_fp8_cache(W.make_tiny(), 64)
    out, lse = run(B, w)
    O, L = ref(w)
    assert_parity(out, lse, O, L, what="fp8 tiny")


@pytest.mark.parametrize("hq,hkv,ps", [(6, 1, 64), (24, 2, 16), (8, 1, 1), (48, 1, 128), (16, 16, 32)])
def test_fp8_multi_tile_ragged(B, hq, hkv, ps):
    w = W.make_chunk(n_rows=96, context=2200, n_qheads=hq, n_kvheads=hkv, topk=2051,
                     seed=hq + 3 * hkv, name="chunk")
    w = W.with_fp8_cache(w, ps)
    out, lse = run(B, w)
    O, L = ref(w)
    assert_parity(out, lse, O, L, what=f"fp8 {hq}/{hkv} page {ps}")


@pytest.mark.parametrize("G", [2, 4])
def test_fp8_union(B, G):
    w = W.with_fp8_cache(W.make_union(n_rows=613, topk=256), 64)
    before = B.counters()
    out, lse = run(B, w, union_g=G)
    assert B.counters()["calls_union"] == before["calls_union"] + 1
    O, L = ref(w)
    assert_parity(out, lse, O, L, what=f"fp8 union G={G}")


def test_fp8_mixed_paged_and_edges(B):
    """Per-row topk_len over a shuffled paged cache, plus rows with no valid slot and slots past
    n_kv_slots."""
    w = W.make_mixed(new_tokens=(64, 150), prefixes=(0, 2000), page_size=64)
    idx = w.indices.copy()
    idx[0] = -1
    idx[3, :40] = w.n_slots + 5
    w = W.with_fp8_cache(W.Workload("mixed", w.q, w.k, w.v, idx, w.topk_len, w.scale, w.positions), 64)
    out, lse = run(B, w, n_kv_slots=w.n_slots)
    O, L = ref(w, n_kv_slots=w.n_slots)
    assert np.isneginf(L[0]).all()
    assert_parity(out, lse, O, L, what="fp8 mixed")


def test_fp8_full_size_group6(B):
    """The group-6 workload with an e4m3 cache (pages of 64), sampled rows against the oracle."""
    w = W.with_fp8_cache(W.make("group6_32k"), 64)
    out, lse = run(B, w)
    rows = np.arange(0, w.n_rows, 331)
    O, L = ref(w, rows=rows)
    assert_parity(out, lse, O, L, rows=rows, what="fp8 group6")
