"""Split items (GPU only): per-token calls with fewer work items than SMs share each item over a
thread-block cluster of 2, 4 or 8 CTAs, each taking a contiguous range of the row's 128-slot
tiles, and merge the partial (max, row sum, O) through distributed shared memory.  The pages
tune the launch shape by row count ("[QSA] Tune sm120 sparse prefill geometry", Query-count
sweep); the result must stay the oracle's.  Bounds: O max-abs 2e-2, LSE relative 1e-3
(helpers.py)."""
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


def ragged(w, seed):
    """Per-row topk_len with the edge cases of a split: no slot, one slot, one tile plus one,
    and the full budget; every fifth slot of one row is padding."""
    rng = np.random.default_rng(seed)
    K = w.indices.shape[1]
    tl = rng.integers(0, K + 1, size=w.n_rows).astype(np.int32)
    special = [0, 1, 129, K]
    if w.n_rows < len(special):
        tl[:] = K
    else:
        tl[:len(special)] = special
    idx = w.indices.copy()
    if w.n_rows > 4:
        idx[4, ::5] = -1
    w.indices, w.topk_len = idx, tl
    return w


def run(B, w, **kw):
    import torch
    q, k, v, idx, tl = to_device(w)
    out, lse = B.sparse_prefill(q, k, v, idx, tl, w.scale, **kw)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    return out, lse


def oracle_full(w):
    return oracle.sparse_prefill(w.q, w.k, w.v, w.indices, w.topk_len, w.scale)


@pytest.mark.parametrize("rows,split", [(1, 8), (7, 8), (33, 4), (64, 2)])
def test_split_rows_match_the_oracle(B, rows, split):
    w = ragged(W.make_chunk(n_rows=rows, context=8192, n_qheads=6, n_kvheads=1, topk=2051,
                            seed=100 + rows, name="split"), rows)
    g = B.select_geometry(6, 1, 0, 2051, 256, rows, 152)
    assert g["split"] == split and g["grid"] == rows * split and g["stages"] == 4
    out, lse = run(B, w)
    O, L = oracle_full(w)
    assert_parity(out, lse, O, L, what=f"split {rows} rows")
    if rows > 1:
        o = out.float().cpu().numpy()
        assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0].cpu().numpy()))   # topk_len 0


@pytest.mark.parametrize("hq,hkv", [(12, 1), (24, 2), (32, 1), (1, 1)])
def test_split_head_shapes(B, hq, hkv):
    w = ragged(W.make_chunk(n_rows=7, context=4000, n_qheads=hq, n_kvheads=hkv, topk=2051,
                            seed=hq + hkv, name="split_heads"), hq)
    out, lse = run(B, w)
    O, L = oracle_full(w)
    assert_parity(out, lse, O, L, what=f"split {hq}/{hkv}")


@pytest.mark.parametrize("forced", [1, 2, 4, 8])
def test_forced_split_agrees_with_unsplit(B, forced):
    """Every split of the same rows (1 = none) matches the oracle; a split of 8 over a 3-tile
    row leaves five CTAs of the cluster with no tile."""
    import torch
    w = ragged(W.make_chunk(n_rows=9, context=3000, n_qheads=6, n_kvheads=1, topk=300,
                            seed=21, name="forced_split"), 21)
    out, lse = run(B, w, forced={"split": forced})
    O, L = oracle_full(w)
    assert_parity(out, lse, O, L, what=f"forced split {forced}")
    ref_out, ref_lse = run(B, w, forced={"split": 1})
    assert float((out.float() - ref_out.float()).abs().max()) <= 2e-2


def test_fp8_small_calls_do_not_split(B):
    """FP8 caches keep one CTA per item (the split is built for bf16 tiles only); a 7-row FP8
    call still matches the FP8 oracle."""
    import torch
    from helpers import compare, O_ATOL, LSE_RTOL
    w = ragged(W.make_chunk(n_rows=7, context=4000, n_qheads=6, n_kvheads=1, topk=2051, seed=31,
                            name="split_fp8"), 31)
    w = W.with_fp8_cache(w, 64)
    m = w.meta
    q, _, _, idx, tl = to_device(w)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out, lse = B.sparse_prefill_fp8(q, t(m["k8"]), t(m["v8"]), t(m["k_scale"]), t(m["v_scale"]),
                                    64, idx, tl, w.scale)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    O, L = oracle.sparse_prefill_fp8_rows(w.q, m["k8"], m["v8"], m["k_scale"], m["v_scale"], 64,
                                          w.indices, w.topk_len, w.scale, np.arange(w.n_rows))
    assert_parity(out, lse, O, L, what="fp8 7 rows")


def test_split_paged(B):
    """Seven rows of a paged batch (logical positions translated in the kernel), split."""
    import torch
    w = W.make_mixed(new_tokens=(3, 2, 1, 1), prefixes=(0, 3000, 700, 5000), page_size=64)
    m = w.meta
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    q, k, v, _, tl = to_device(w)
    out, lse = B.sparse_prefill_paged(q, k, v, i32(m["logical_indices"]), tl,
                                      i32(m["cu_seqlens_q"]), i32(m["kv_lens_array"]),
                                      i32(m["page_table"]), 64, w.scale, n_pages=m["n_pages"])
    torch.cuda.synchronize()
    assert B.device_status() == 0
    O, L = oracle_full(w)
    assert_parity(out, lse, O, L, what="split paged")


def test_split_noalloc_graph_and_determinism(B):
    import torch
    w = ragged(W.make_chunk(n_rows=5, context=6000, n_qheads=6, n_kvheads=1, topk=2051, seed=41,
                            name="split_graph"), 41)
    q, k, v, idx, tl = to_device(w)
    o1, l1 = B.sparse_prefill(q, k, v, idx, tl, w.scale)
    o2, l2 = B.sparse_prefill_noalloc(q, k, v, idx, tl, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)
    out = torch.zeros_like(q)
    lse = torch.zeros_like(l1)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.sparse_prefill(q, k, v, idx, tl, w.scale, out=out, lse=lse)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), o1.view(torch.int16)) and torch.equal(lse, l1)
    O, L = oracle_full(w)
    assert_parity(o1, l1, O, L, what="split 5 rows")
