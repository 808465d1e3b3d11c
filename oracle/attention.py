"""Per-token sparse attention prefill, float64, the plain definition.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Definition (pages: "[QSA] Tune sm120 sparse prefill geometry", Motivation and
Tests; "DSA prefill ... triton_sparse_mla", Motivation and Robustness):

    for row r, query head h:
        kvh   = h // g                       g = n_qheads // n_kvheads
        L     = topk if topk_len is None else clamp(topk_len[r], 0, topk)
        J     = [ idx[r, j] for j < L if idx[r, j] >= 0
                  and (n_kv_slots == 0 or idx[r, j] < n_kv_slots) ]   (a multiset)
        s_j   = scale * <q[r, h, :], K[J_j, kvh, :]>
        O     = sum_j exp(s_j - m) V[J_j, kvh, :] / sum_j exp(s_j - m),  m = max_j s_j
        LSE   = m + ln sum_j exp(s_j - m)         (natural log of the scaled logits)
        empty J: O = 0, LSE = -inf

Readings where the pages are silent: every negative index is padding (not
only -1); an index >= n_kv_slots is padding when the slot count is given;
``topk_len`` counts leading slots; a slot listed twice is weighted twice;
query head h reads KV head h // g; one index row serves every KV head.
"""
from __future__ import annotations

import numpy as np


def _bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact widening)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _as_f64(x: np.ndarray) -> np.ndarray:
    """Accept raw bf16 bits (uint16) or any float array."""
    if x.dtype == np.uint16:
        return _bf16_bits_to_f64(x)
    return np.asarray(x, dtype=np.float64)


def valid_slots(index_row: np.ndarray, topk_len_r, n_kv_slots: int = 0) -> np.ndarray:
    """Selected slots of one row that take part, in slot order (duplicates kept)."""
    topk = index_row.shape[0]
    L = topk if topk_len_r is None else int(min(max(int(topk_len_r), 0), topk))
    sel = np.asarray(index_row[:L], dtype=np.int64)
    keep = sel >= 0
    if n_kv_slots > 0:
        keep &= sel < n_kv_slots
    return sel[keep]


def _attend(qg: np.ndarray, ksel: np.ndarray, vsel: np.ndarray, scale: float):
    """qg [g, D], ksel [n, D], vsel [n, Dv] -> (O [g, Dv], lse [g]) in float64."""
    g = qg.shape[0]
    if ksel.shape[0] == 0:                       # no valid slot: O = 0, LSE = -inf
        return np.zeros((g, vsel.shape[1])), np.full(g, -np.inf)
    s = scale * (qg @ ksel.T)                    # [g, n]
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=1, keepdims=True)
    O = (p @ vsel) / l
    lse = (m + np.log(l))[:, 0]
    return O, lse


def sparse_prefill_rows(q, k, v, indices, topk_len, scale, rows, n_kv_slots: int = 0):
    """Oracle O / LSE for the listed rows only.

    q [R, Hq, D], k/v [S, Hkv, D] (bf16 bits or floats), indices [R, topk] int.
    Returns O [len(rows), Hq, D] float64 and LSE [len(rows), Hq] float64.
    """
    R, Hq, D = q.shape
    Hkv = k.shape[1]
    if Hq % Hkv != 0:
        raise ValueError("n_qheads must be a multiple of n_kvheads")
    g = Hq // Hkv
    rows = np.asarray(rows, dtype=np.int64)
    O = np.zeros((len(rows), Hq, D))
    lse = np.full((len(rows), Hq), -np.inf)
    for i, r in enumerate(rows):
        tl = None if topk_len is None else topk_len[r]
        J = valid_slots(indices[r], tl, n_kv_slots)
        qr = _as_f64(q[r])                       # [Hq, D]
        for kvh in range(Hkv):
            ksel = _as_f64(k[J, kvh, :]) if len(J) else np.zeros((0, D))
            vsel = _as_f64(v[J, kvh, :]) if len(J) else np.zeros((0, D))
            hs = slice(kvh * g, (kvh + 1) * g)
            O[i, hs], lse[i, hs] = _attend(qr[hs], ksel, vsel, scale)
    return O, lse


def sparse_prefill(q, k, v, indices, topk_len, scale, n_kv_slots: int = 0):
    """Oracle O [R, Hq, D] and LSE [R, Hq] (float64) for every row."""
    return sparse_prefill_rows(q, k, v, indices, topk_len, scale,
                               np.arange(q.shape[0]), n_kv_slots)
