"""Sparse attention prefill over a paged KV cache with ragged request metadata, float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Pages: "DSA prefill ... triton_sparse_mla" (Modifications, Robustness: a batch's top-k indices go
through a PAGED or a RAGGED transform chosen per batch kind, and the valid length comes from the
cache sequence lengths; the review follow-up on MIXED batches) and "[QSA] Tune sm120 sparse
prefill geometry" (the serving command's paged cache, --page-size 128).

Definition (the pages leave the page arithmetic implicit; this is the plain reading):

    row r belongs to request i, the last i with cu_seqlens_q[i] <= r
    position x of row r is padding if x < 0, x >= kv_lens[i] (when given),
        x // page_size >= pages_per_req, or the page id
        pid = page_table[i, x // page_size] is < 0 or >= n_pages (when n_pages > 0);
    otherwise it reads physical slot pid * page_size + x % page_size.

The attention over the resulting physical slots is ``attention.sparse_prefill`` unchanged
(topk_len counts leading positions of the row, before translation).
"""
from __future__ import annotations

import numpy as np

from .attention import sparse_prefill_rows


def request_of_rows(cu_seqlens_q: np.ndarray, n_rows: int) -> np.ndarray:
    """Request index of every row: the last request whose first row is <= the row."""
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    req = np.zeros(n_rows, dtype=np.int64)
    for r in range(n_rows):
        i = 0
        for cand in range(len(cu) - 1):
            if cu[cand] <= r:
                i = cand
        req[r] = i
    return req


def physical_indices(indices, cu_seqlens_q, kv_lens, page_table, page_size: int,
                     n_pages: int = 0) -> np.ndarray:
    """Logical positions [R, topk] -> physical slots [R, topk] (int64, -1 = padding)."""
    idx = np.asarray(indices, dtype=np.int64)
    R, K = idx.shape
    table = np.asarray(page_table, dtype=np.int64)
    pages_per_req = table.shape[1]
    req = request_of_rows(cu_seqlens_q, R)
    out = np.full((R, K), -1, dtype=np.int64)
    for r in range(R):
        i = req[r]
        x = idx[r]
        kv_len = np.iinfo(np.int64).max if kv_lens is None else int(kv_lens[i])
        page = np.where(x >= 0, x // page_size, 0)
        ok = (x >= 0) & (x < kv_len) & (page < pages_per_req)
        pid = np.where(ok, table[i, np.minimum(page, pages_per_req - 1)], -1)
        ok &= pid >= 0
        if n_pages > 0:
            ok &= pid < n_pages
        out[r] = np.where(ok, pid * page_size + x % page_size, -1)
    return out


def sparse_prefill_paged_rows(q, k_cache, v_cache, indices, topk_len, cu_seqlens_q, kv_lens,
                              page_table, page_size: int, scale: float, rows,
                              n_pages: int = 0):
    """Oracle O / LSE for the listed rows of a paged call."""
    rows = np.asarray(rows, dtype=np.int64)
    phys = physical_indices(indices, cu_seqlens_q, kv_lens, page_table, page_size, n_pages)
    return sparse_prefill_rows(q, k_cache, v_cache, phys, topk_len, scale, rows)


def sparse_prefill_paged(q, k_cache, v_cache, indices, topk_len, cu_seqlens_q, kv_lens,
                         page_table, page_size: int, scale: float, n_pages: int = 0):
    """Oracle O [R, Hq, D] and LSE [R, Hq] (float64) for every row of a paged call."""
    return sparse_prefill_paged_rows(q, k_cache, v_cache, indices, topk_len, cu_seqlens_q,
                                     kv_lens, page_table, page_size, scale,
                                     np.arange(q.shape[0]), n_pages)
