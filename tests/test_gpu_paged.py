"""qsa_sparse_prefill_paged (logical positions + page table, translated in the kernels) against
the paged oracle, and bit for bit against the plain entry given the same batch's physical slots
(GPU only).  Both entries compact the same slots in the same order, so their arithmetic is
identical."""
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


def i32(a):
    import torch
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def paged_call(B, w, logical, cu, kv_lens, table, page_size, n_pages=0, union_g=0):
    import torch
    q, k, v, _, tl = to_device(w)
    out, lse = B.sparse_prefill_paged(q, k, v, i32(logical), tl, i32(cu), i32(kv_lens), i32(table),
                                      page_size, w.scale, n_pages=n_pages, union_g=union_g)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    return out, lse


def paged_oracle(w, logical, cu, kv_lens, table, page_size, n_pages=0, rows=None):
    rows = np.arange(w.n_rows) if rows is None else rows
    return oracle.sparse_prefill_paged_rows(w.q, w.k, w.v, logical, w.topk_len, cu, kv_lens, table,
                                            page_size, w.scale, rows, n_pages)


def small_mixed(**kw):
    return W.make_mixed(new_tokens=kw.get("new", (64, 200, 130, 300)),
                        prefixes=kw.get("pre", (0, 3000, 700, 5000)),
                        page_size=kw.get("ps", 64), topk=kw.get("topk", 2051))


@pytest.mark.parametrize("union_g", [0, 2, 4])
def test_paged_small_matches_oracle_and_plain_entry(B, union_g):
    import torch
    w = small_mixed()
    m = w.meta
    out, lse = paged_call(B, w, m["logical_indices"], m["cu_seqlens_q"], m["kv_lens_array"],
                          m["page_table"], m["page_size"], m["n_pages"], union_g)
    O, L = paged_oracle(w, m["logical_indices"], m["cu_seqlens_q"], m["kv_lens_array"],
                        m["page_table"], m["page_size"], m["n_pages"])
    assert_parity(out, lse, O, L, what=f"paged G={union_g}")
    q, k, v, idx, tl = to_device(w)
    out2, lse2 = B.sparse_prefill(q, k, v, idx, tl, w.scale, union_g=union_g)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse, lse2)


@pytest.mark.parametrize("page_size", [1, 16, 48, 128])
def test_paged_page_sizes_and_no_kv_lens(B, page_size):
    """Power-of-two and other page sizes; kv_lens absent (pages bound the request) and
    n_pages unchecked."""
    w = small_mixed(ps=page_size, new=(40, 90), pre=(500, 1200), topk=700)
    m = w.meta
    out, lse = paged_call(B, w, m["logical_indices"], m["cu_seqlens_q"], None, m["page_table"],
                          page_size)
    O, L = paged_oracle(w, m["logical_indices"], m["cu_seqlens_q"], None, m["page_table"],
                        page_size)
    assert_parity(out, lse, O, L, what=f"page size {page_size}")


def test_paged_padding_rules(B):
    """Empty requests (repeated offsets), positions past kv_len, past the page-table row and on
    missing or out-of-range pages, negative positions: all padding, including whole rows."""
    rng = np.random.default_rng(91)
    w = small_mixed(new=(30, 50, 20), pre=(600, 100, 900), ps=32, topk=400)
    m = w.meta
    logical = m["logical_indices"].copy()
    cu = m["cu_seqlens_q"]
    # insert two empty requests: request ids shift, the table and kv_lens grow to match
    cu2 = np.array([0, 0, cu[1], cu[2], cu[2], cu[3]], dtype=np.int32)
    table = m["page_table"]
    t2 = np.full((5, table.shape[1] + 2), -1, dtype=np.int32)
    t2[1, :table.shape[1]] = table[0]
    t2[2, :table.shape[1]] = table[1]
    t2[4, :table.shape[1]] = table[2]
    kvl = m["kv_lens_array"]
    kvl2 = np.array([0, kvl[0], kvl[1] - 7, 0, kvl[2]], dtype=np.int32)   # request 2 shortened
    n_pages = m["n_pages"]
    t2[4, 3] = n_pages + 5                               # out of range: padding when checked
    t2[1, 2] = -1                                        # missing page
    R = logical.shape[0]
    for r in range(R):                                   # junk past every limit
        logical[r, rng.integers(0, 400, 5)] = rng.integers(t2.shape[1] * 32, t2.shape[1] * 32 + 99, 5)
        logical[r, rng.integers(0, 400, 3)] = -rng.integers(1, 9, 3)
    logical[5, :] = -1                                   # a row with nothing valid
    out, lse = paged_call(B, w, logical, cu2, kvl2, t2, 32, n_pages)
    O, L = paged_oracle(w, logical, cu2, kvl2, t2, 32, n_pages)
    assert np.isneginf(L[5]).all()
    assert_parity(out, lse, O, L, what="paged padding rules")


def test_paged_many_requests(B):
    """300 requests of 1-9 rows: the request lookup takes two rounds of the 32-ary search."""
    rng = np.random.default_rng(92)
    n_req, ps, topk, Hq = 300, 16, 96, 6
    rows = rng.integers(1, 10, n_req)
    kv = rng.integers(20, 400, n_req)
    pages = -(-kv // ps)
    n_pages = int(pages.sum())
    perm = rng.permutation(n_pages)
    table = np.full((n_req, int(pages.max())), -1, dtype=np.int32)
    off = 0
    for i in range(n_req):
        table[i, :pages[i]] = perm[off:off + pages[i]]
        off += pages[i]
    R = int(rows.sum())
    cu = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    logical = np.full((R, topk), -1, dtype=np.int32)
    r = 0
    for i in range(n_req):
        for _ in range(rows[i]):
            n = min(topk, int(kv[i]))
            logical[r, :n] = rng.choice(int(kv[i]), n, replace=False)
            r += 1
    q = W.randn_bf16(rng, (R, Hq, 256))
    k = W.randn_bf16(rng, (n_pages * ps, 1, 256))
    v = W.randn_bf16(rng, (n_pages * ps, 1, 256))
    w = W.Workload("many_requests", q, k, v, logical, None, 1.0 / 16.0, np.zeros(R, np.int64))
    out, lse = paged_call(B, w, logical, cu, kv.astype(np.int32), table, ps, n_pages)
    O, L = paged_oracle(w, logical, cu, kv, table, ps, n_pages)
    assert_parity(out, lse, O, L, what="300 requests")


def test_paged_full_size_mixed_batch(B, oracle_pool):
    """The chunked mixed batch (4 requests, 14848 rows, 2024 pages of 64) through the paged
    entry: bit-identical to the plain entry on the translated slots, and every row against the
    paged oracle."""
    import torch
    w = W.make("mixed_paged")
    m = w.meta
    out, lse = paged_call(B, w, m["logical_indices"], m["cu_seqlens_q"], m["kv_lens_array"],
                          m["page_table"], m["page_size"], m["n_pages"])
    q, k, v, idx, tl = to_device(w)
    out2, lse2 = B.sparse_prefill(q, k, v, idx, tl, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse, lse2)
    oracle_pool.check_all_rows(("mixed_paged", ""), "paged", out, lse, "full mixed batch, paged entry")
