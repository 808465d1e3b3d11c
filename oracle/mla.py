"""Sparse attention prefill in the MLA shape, float64, the plain definition.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Pages: "DSA prefill ... triton_sparse_mla" (Motivation: GLM-5.x DSA prefill at TP8, 8 real heads;
Speed Tests: kv_lora_rank 512 + qk_rope_head_dim 64 = 576, d_v 512, topk 2048).  Each slot holds
one latent row shared by every head; its 576 dims are the key, its first 512 dims the value:

    for row r, head h:
        J   = valid slots of row r (as attention.valid_slots: topk_len, negative = padding,
              slot >= n_kv_slots = padding when the count is given; duplicates kept)
        s_j = scale * <q[r, h, :576], kv[J_j, :576]>
        O   = sum_j softmax(s)_j kv[J_j, :512],   LSE = ln sum_j exp(s_j)
        empty J: O = 0, LSE = -inf
"""
from __future__ import annotations

import numpy as np

from .attention import _as_f64, _attend, valid_slots


def sparse_mla_prefill_rows(q, kv, indices, topk_len, scale: float, rows, d_v: int = 512,
                            n_kv_slots: int = 0):
    """q [R, H, d_qk], kv [S, d_qk] (bf16 bits or floats), indices [R, topk].
    Returns O [len(rows), H, d_v] and LSE [len(rows), H] in float64."""
    R, H, Dqk = q.shape
    if kv.shape[-1] != Dqk or d_v > Dqk:
        raise ValueError("kv rows must have d_qk dims and d_v <= d_qk")
    kv2 = kv.reshape(kv.shape[0], Dqk)
    rows = np.asarray(rows, dtype=np.int64)
    O = np.zeros((len(rows), H, d_v))
    lse = np.full((len(rows), H), -np.inf)
    for i, r in enumerate(rows):
        tl = None if topk_len is None else topk_len[r]
        J = valid_slots(indices[r], tl, n_kv_slots)
        rows_kv = _as_f64(kv2[J]) if len(J) else np.zeros((0, Dqk))
        O[i], lse[i] = _attend(_as_f64(q[r]), rows_kv, rows_kv[:, :d_v], scale)
    return O, lse


def sparse_mla_prefill(q, kv, indices, topk_len, scale: float, d_v: int = 512,
                       n_kv_slots: int = 0):
    """Oracle O [R, H, d_v] and LSE [R, H] (float64) for every row."""
    return sparse_mla_prefill_rows(q, kv, indices, topk_len, scale, np.arange(q.shape[0]), d_v,
                                   n_kv_slots)
