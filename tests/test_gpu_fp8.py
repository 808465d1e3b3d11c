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


@pytest.mark.parametrize("G", [0, 4])
def test_fp8_full_size(B, oracle_pool, G):
    """The group-6 workload (per-token) and the union workload (G = 4) with e4m3 caches (pages of
    64), every row against the FP8 oracle."""
    name = "group6_32k" if G == 0 else "union_8k"
    w = W.with_fp8_cache(W.make(name), 64)
    out, lse = run(B, w, union_g=G)
    oracle_pool.check_all_rows((name, "fp8:64"), "fp8", out, lse, f"fp8 {name} G={G}")


@pytest.mark.parametrize("c", [4096.0, 3.0e4, 1.0e-6])
def test_fp8_large_and_small_v_scales(B, c):
    """V page scales multiplied by c: O scales by c exactly and LSE is unchanged.  With c = 3e4 a
    probability times its V scale passes the fp16 range unless the kernel normalises the scales
    per item; with c = 1e-6 it would fall into fp16 subnormals."""
    from helpers import compare, O_ATOL, LSE_RTOL
    w = W.with_fp8_cache(W.make_chunk(n_rows=64, context=3000, n_qheads=6, n_kvheads=1, topk=2051,
                                      seed=77, name="vscale"), 64)
    w.meta["v_scale"] = (w.meta["v_scale"] * np.float32(c)).astype(np.float32)
    out, lse = run(B, w)
    O, L = ref(w)
    dO, dL, mism = compare(out.float() / c, lse, O / c, L)
    assert mism == 0 and dO <= O_ATOL and dL <= LSE_RTOL, (c, dO, dL, mism)


def test_fp8_mixed_page_scale_magnitudes(B):
    """Per-page V scales spread over four decades and K scales over one, union and per-token:
    errors stay within 2e-2 of the largest output magnitude."""
    from helpers import compare, LSE_RTOL
    rng = np.random.default_rng(78)
    for G in (0, 2):
        w = W.with_fp8_cache(W.make_union(n_rows=300, topk=384), 16)
        m = w.meta
        m["v_scale"] = (m["v_scale"] * 10.0 ** rng.uniform(-2, 2, m["v_scale"].shape)).astype(np.float32)
        m["k_scale"] = (m["k_scale"] * 10.0 ** rng.uniform(-0.5, 0.5, m["k_scale"].shape)).astype(np.float32)
        out, lse = run(B, w, union_g=G)
        O, L = ref(w)
        dO, dL, mism = compare(out, lse, O, L)
        bound = 2e-2 * max(1.0, float(np.abs(O).max()))
        assert mism == 0 and dO <= bound and dL <= LSE_RTOL, (G, dO, bound, dL, mism)


@pytest.mark.parametrize("G", [0, 4])
def test_fp8_paged_matches_oracle_and_plain_fp8_entry(B, G):
    """FP8 caches over a paged pool: logical indices translated in the kernels, e4m3 scales by
    physical slot.  Against the FP8 oracle on the batch's physical slots, and bit for bit against
    the plain FP8 entry given those slots (both compact the same slots in the same order)."""
    import torch
    w = W.make_mixed(new_tokens=(64, 200, 130, 300), prefixes=(0, 3000, 700, 5000), page_size=64)
    w = W.with_fp8_cache(w, 16)                  # scale pages of 16 slots, pool pages of 64
    m = w.meta
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    q, _, _, idx, tl = to_device(w)
    out, lse = B.sparse_prefill_fp8_paged(q, t(m["k8"]), t(m["v8"]), t(m["k_scale"]), t(m["v_scale"]),
                                          16, i32(m["logical_indices"]), tl, i32(m["cu_seqlens_q"]),
                                          i32(m["kv_lens_array"]), i32(m["page_table"]), 64, w.scale,
                                          n_pages=m["n_pages"], union_g=G)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    O, L = ref(w)
    assert_parity(out, lse, O, L, what=f"fp8 paged G={G}")
    out2, lse2 = B.sparse_prefill_fp8(q, t(m["k8"]), t(m["v8"]), t(m["k_scale"]), t(m["v_scale"]),
                                      16, idx, tl, w.scale, union_g=G)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse, lse2)
