"""G-token union of selected slots with a per-row ownership bitmask.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows "DSA prefill ... triton_sparse_mla", Modifications: G adjacent query
rows share one gathered index set.  Every row's selection is sorted by itself;
a slot enters the group's list through the first row that selected it, and its
ownership bits record every row of the group whose selection holds it.  The
Accuracy Tests section of that page states the resulting contract: a slot is
listed once per group, its bits are the OR over the rows that own it, and -1
padding never appears.

Readings (the page prints no layout):
* groups are G consecutive rows of the flat row array; the last group may
  hold G' < G rows;
* list order is canonical: row 0's emitted slots ascending, then row 1's, ...;
* bit u of ``union_bits`` (uint8) is row u of the group, so G <= 8;
* a row's valid set applies the same filter as the per-token path (topk_len,
  negative indices, slots >= n_kv_slots when given); a slot repeated inside
  one row is listed once;
* lists are padded with -1 to G * topk entries, bits with 0;
  ``union_len`` is the emitted count.
* ``sorted_rows`` returns each row's valid slots ascending (repeats kept),
  then -1.
"""
from __future__ import annotations

import numpy as np

from .attention import valid_slots, _attend, _as_f64


def sorted_rows(indices: np.ndarray, topk_len, n_kv_slots: int = 0) -> np.ndarray:
    R, K = indices.shape
    out = np.full((R, K), -1, dtype=np.int32)
    for r in range(R):
        tl = None if topk_len is None else topk_len[r]
        J = np.sort(valid_slots(indices[r], tl, n_kv_slots))
        out[r, :len(J)] = J
    return out


def union_build(indices: np.ndarray, topk_len, G: int, n_kv_slots: int = 0):
    """Returns (union_idx [n_groups, G*K] int32, union_bits [n_groups, G*K] uint8,
    union_len [n_groups] int32)."""
    if not (1 <= G <= 8):
        raise ValueError("G must be in [1, 8]")
    R, K = indices.shape
    n_groups = -(-R // G)
    uidx = np.full((n_groups, G * K), -1, dtype=np.int32)
    ubits = np.zeros((n_groups, G * K), dtype=np.uint8)
    ulen = np.zeros(n_groups, dtype=np.int32)
    for gi in range(n_groups):
        rows = range(gi * G, min((gi + 1) * G, R))
        sets = []
        for r in rows:
            tl = None if topk_len is None else topk_len[r]
            sets.append(np.unique(valid_slots(indices[r], tl, n_kv_slots)))  # sorted, distinct
        n = 0
        for t, St in enumerate(sets):
            earlier = np.concatenate(sets[:t]) if t else np.zeros(0, dtype=np.int64)
            emit = St[~np.isin(St, earlier)]
            bits = np.zeros(len(emit), dtype=np.uint8)
            for u, Su in enumerate(sets):
                bits |= (np.isin(emit, Su).astype(np.uint8) << np.uint8(u))
            uidx[gi, n:n + len(emit)] = emit
            ubits[gi, n:n + len(emit)] = bits
            n += len(emit)
        ulen[gi] = n
    return uidx, ubits, ulen


def union_attention(q, k, v, union_idx, union_bits, union_len, G: int, scale: float):
    """O / LSE of every row computed from its group's union list, keeping only the
    entries whose ownership bit for that row is set."""
    R, Hq, D = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    O = np.zeros((R, Hq, D))
    lse = np.full((R, Hq), -np.inf)
    for r in range(R):
        gi, u = divmod(r, G)
        n = int(union_len[gi])
        lst = np.asarray(union_idx[gi, :n], dtype=np.int64)
        own = (union_bits[gi, :n] >> np.uint8(u)) & np.uint8(1)
        J = lst[own.astype(bool)]
        qr = _as_f64(q[r])
        for kvh in range(Hkv):
            hs = slice(kvh * g, (kvh + 1) * g)
            ksel = _as_f64(k[J, kvh, :]) if len(J) else np.zeros((0, D))
            vsel = _as_f64(v[J, kvh, :]) if len(J) else np.zeros((0, D))
            O[r, hs], lse[r, hs] = _attend(qr[hs], ksel, vsel, scale)
    return O, lse
