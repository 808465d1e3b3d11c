"""CUDA path vs the CPU oracle, element by element, on seeded synthetic inputs (GPU only).

Small cases cover several 128-slot tiles and a ragged tail and are compared in full; the
full-size workloads are run exactly as the benchmark launches them and compared on sampled
rows.  Bounds: O max-abs 2e-2, LSE relative 1e-3 (see helpers.py)."""
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


def run(B, w, union_g=0, **kw):
    q, k, v, idx, tl = to_device(w)
    out, lse = B.sparse_prefill(q, k, v, idx, tl, w.scale, union_g=union_g, **kw)
    import torch
    torch.cuda.synchronize()
    assert B.device_status() == 0
    return out, lse


def oracle_full(w, **kw):
    return oracle.sparse_prefill(w.q, w.k, w.v, w.indices, w.topk_len, w.scale, **kw)


def test_tiny_config_full(B):
    w = W.make_tiny()
    out, lse = run(B, w)
    O, L = oracle_full(w)
    assert_parity(out, lse, O, L, what="tiny")


@pytest.mark.parametrize("hq,hkv", [(6, 1), (12, 1), (24, 2), (8, 1), (1, 1), (16, 16)])
def test_chunk_multi_tile_ragged(B, hq, hkv):
    # 2051 slots = 16 full tiles + a 3-slot tail; rows near the start have short prefixes
    w = W.make_chunk(n_rows=160, context=2200, n_qheads=hq, n_kvheads=hkv, topk=2051,
                     seed=hq * 7 + hkv, name="chunk")
    out, lse = run(B, w)
    O, L = oracle_full(w)
    assert_parity(out, lse, O, L, what=f"chunk {hq}/{hkv}")


@pytest.mark.parametrize("topk", [1, 7, 127, 128, 129, 300, 1000])
def test_topk_widths(B, topk):
    w = W.make_chunk(n_rows=70, context=1500, n_qheads=6, n_kvheads=1, topk=topk, seed=topk,
                     name="widths")
    out, lse = run(B, w)
    O, L = oracle_full(w)
    assert_parity(out, lse, O, L, what=f"topk {topk}")


def test_mixed_paged_small(B):
    w = W.make_mixed(new_tokens=(64, 200, 130, 300), prefixes=(0, 3000, 700, 5000), page_size=64)
    out, lse = run(B, w)
    O, L = oracle_full(w)
    assert_parity(out, lse, O, L, what="mixed paged")


def test_edge_rows(B):
    """All -1 rows, topk_len = 0, negative indices other than -1, duplicates (weighted twice),
    junk past topk_len."""
    rng = np.random.default_rng(77)
    R, S, K = 12, 600, 300
    w = W.make_chunk(n_rows=R, context=S, n_qheads=6, n_kvheads=1, topk=K, seed=5, name="edge")
    idx = w.indices.copy()
    tl = np.full(R, K, dtype=np.int32)
    idx[0] = -1                                  # no valid slot
    tl[1] = 0                                    # topk_len 0
    idx[2, ::3] = -5                             # other negative values are padding
    idx[3, 1] = idx[3, 0]                        # a repeated slot counts twice
    idx[3, 2] = idx[3, 0]
    tl[4] = 37
    idx[4, 37:] = rng.integers(0, S, size=K - 37)   # junk past topk_len
    tl[5] = 1
    idx[6, :] = -1
    idx[6, K - 1] = 17                           # only the last slot is valid
    w.indices, w.topk_len = idx, tl
    out, lse = run(B, w)
    O, L = oracle_full(w)
    assert_parity(out, lse, O, L, what="edge rows")
    o = out.float().cpu().numpy()
    assert np.all(o[0] == 0) and np.all(o[1] == 0)
    assert np.all(np.isneginf(lse[0].cpu().numpy())) and np.all(np.isneginf(lse[1].cpu().numpy()))


def test_out_of_range_slots_with_slot_count(B):
    w = W.make_chunk(n_rows=40, context=900, n_qheads=6, n_kvheads=1, topk=400, seed=9, name="oor")
    idx = w.indices.copy()
    idx[:, ::7] = 900 + np.arange(idx[:, ::7].shape[1])[None, :]   # >= n_kv_slots: padding
    w.indices = idx
    out, lse = run(B, w, n_kv_slots=900)
    O, L = oracle_full(w, n_kv_slots=900)
    assert_parity(out, lse, O, L, what="slot-count filter")


def test_single_row_and_lse_optional(B):
    import torch
    w = W.make_chunk(n_rows=1, context=3000, n_qheads=6, n_kvheads=1, topk=2051, seed=3, name="one")
    q, k, v, idx, tl = to_device(w)
    out, _ = B.sparse_prefill(q, k, v, idx, tl, w.scale, want_lse=False)
    torch.cuda.synchronize()
    O, L = oracle_full(w)
    assert float(np.max(np.abs(out.float().cpu().numpy() - O))) <= 2e-2


def test_deterministic_and_side_stream(B):
    import torch
    w = W.make_chunk(n_rows=300, context=5000, n_qheads=6, n_kvheads=1, topk=2051, seed=11, name="det")
    q, k, v, idx, tl = to_device(w)
    o1, l1 = B.sparse_prefill(q, k, v, idx, tl, w.scale)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o2, l2 = B.sparse_prefill(q, k, v, idx, tl, w.scale)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_cuda_graph_replay(B):
    import torch
    w = W.make_chunk(n_rows=200, context=3000, n_qheads=6, n_kvheads=1, topk=2051, seed=12, name="graph")
    q, k, v, idx, tl = to_device(w)
    out = torch.empty_like(q)
    lse = torch.empty((w.n_rows, w.n_qheads), dtype=torch.float32, device="cuda")
    B.sparse_prefill(q, k, v, idx, tl, w.scale, out=out, lse=lse)     # warm-up outside capture
    torch.cuda.synchronize()
    ref = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.sparse_prefill(q, k, v, idx, tl, w.scale, out=out, lse=lse)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_counters_and_step_down(B):
    import torch
    w = W.make_chunk(n_rows=50, context=2500, n_qheads=6, n_kvheads=1, topk=2051, seed=13, name="cnt")
    q, k, v, idx, tl = to_device(w)
    B.reset_counters()
    B.sparse_prefill(q, k, v, idx, tl, w.scale)
    out, lse = B.sparse_prefill(q, k, v, idx, tl, w.scale, forced={"stages": 16, "grid": 7})
    torch.cuda.synchronize()
    c = B.counters()
    assert c["calls_per_token"] == 2 and c["step_downs"] == 1 and c["kernel_launches"] == 2
    O, L = oracle_full(w)
    assert_parity(out, lse, O, L, what="forced geometry")
