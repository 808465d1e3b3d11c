"""Checks that pin the CPU oracle to facts outside the oracle itself.

Each ``check_*`` takes an attention callable with the oracle's signature
``fn(q, k, v, indices, topk_len, scale, n_kv_slots=0) -> (O, LSE)`` (or a
union-build callable) and returns a list of failure messages (empty = pass).
``test_oracle_pins.py`` runs them on the oracle; ``test_oracle_mutants.py``
runs them on copies of the oracle with one planted mistake each and requires
that some check fails, so the pins are known to bite.

Independent facts used:
* dense causal GQA attention from torch's CPU flash-attention routine
  (output and log-sum-exp) -- sparse attention over the whole causal prefix
  must equal it ("DSA prefill ... triton_sparse_mla", Speed Tests: below the
  dense-threshold the dense one-shot path is interchangeable);
* scipy's logsumexp and numpy's mean for closed forms (zero query, one slot,
  identical keys);
* invariances under slot permutation, inserted padding, topk_len truncation,
  the slot-count filter and KV-head replication;
* hand-derived golden cases (tests/golden/hand_cases.json);
* brute-force Python set arithmetic for the union contract.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch
from scipy.special import logsumexp

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _close(a, b, tol):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.shape != b.shape:
        return False
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        diff = np.where(both_inf, 0.0, np.abs(a - b))
    return bool(np.all(np.isfinite(diff)) and diff.max(initial=0.0) <= tol)


def _rng(seed):
    return np.random.default_rng(seed)


def dense_case(seed=0, S=40, R=20, Hq=6, Hkv=2, D=16, topk=48, scale=0.37):
    """Rows at positions S-R..S-1 whose selection is their whole causal prefix, shuffled."""
    rng = _rng(seed)
    q = rng.standard_normal((R, Hq, D))
    k = rng.standard_normal((S, Hkv, D))
    v = rng.standard_normal((S, Hkv, D))
    pos = np.arange(S - R, S)
    idx = np.full((R, topk), -1, dtype=np.int32)
    for r, p in enumerate(pos):
        perm = rng.permutation(p + 1)
        slots = rng.choice(topk, size=p + 1, replace=False)   # scatter among -1 padding
        idx[r, slots] = perm
    return q, k, v, idx, pos, scale


def dense_reference(q, k, v, pos, scale):
    """torch CPU flash attention (float64), causal by absolute position, GQA by h // g."""
    R, Hq, D = q.shape
    S, Hkv, _ = k.shape
    g = Hq // Hkv
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]                          # [1, Hq, R, D]
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(g, dim=0)[None]
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(g, dim=0)[None]
    mask = torch.zeros((1, 1, R, S), dtype=torch.float64)
    keypos = torch.arange(S)[None, :]
    mask[0, 0] = torch.where(keypos <= torch.from_numpy(pos)[:, None], 0.0, float("-inf"))
    out, lse = torch.ops.aten._scaled_dot_product_flash_attention_for_cpu(
        tq, tk, tv, 0.0, False, attn_mask=mask, scale=scale)
    return out[0].permute(1, 0, 2).numpy(), lse[0].permute(1, 0).numpy()


def check_dense_equivalence(fn):
    fails = []
    for seed, (Hq, Hkv) in enumerate([(6, 2), (6, 1), (4, 4), (8, 2)]):
        q, k, v, idx, pos, scale = dense_case(seed=seed, Hq=Hq, Hkv=Hkv)
        O, L = fn(q, k, v, idx, None, scale)
        Od, Ld = dense_reference(q, k, v, pos, scale)
        if not _close(O, Od, 1e-10):
            fails.append(f"dense O mismatch (Hq={Hq}, Hkv={Hkv})")
        if not _close(L, Ld, 1e-10):
            fails.append(f"dense LSE mismatch (Hq={Hq}, Hkv={Hkv})")
    return fails


def check_zero_query(fn):
    """q = 0: every logit is 0, so O = mean of the selected V rows, LSE = ln(count)."""
    rng = _rng(11)
    S, Hkv, D, R, K = 30, 1, 8, 5, 12
    q = np.zeros((R, 3, D))
    k = rng.standard_normal((S, Hkv, D))
    v = rng.standard_normal((S, Hkv, D))
    idx = np.full((R, K), -1, dtype=np.int32)
    counts = [1, 3, 7, 12, 5]
    for r, n in enumerate(counts):
        idx[r, :n] = rng.choice(S, size=n, replace=False)
    O, L = fn(q, k, v, idx, None, 0.5)
    fails = []
    for r, n in enumerate(counts):
        want = np.mean(v[idx[r, :n], 0, :], axis=0)
        if not _close(O[r], np.broadcast_to(want, O[r].shape), 1e-12):
            fails.append(f"zero-query O row {r}")
        if not _close(L[r], np.full(3, math.log(n)), 1e-12):
            fails.append(f"zero-query LSE row {r}")
    return fails


def check_single_slot(fn):
    """One valid slot: O is that V row exactly, LSE is its scaled logit."""
    rng = _rng(12)
    S, D = 9, 8
    q = rng.standard_normal((1, 2, D))
    k = rng.standard_normal((S, 1, D))
    v = rng.standard_normal((S, 1, D))
    idx = np.array([[-1, 4, -1, -1]], dtype=np.int32)
    scale = 0.8
    O, L = fn(q, k, v, idx, None, scale)
    fails = []
    for h in range(2):
        s = scale * math.fsum(float(a) * float(b) for a, b in zip(q[0, h], k[4, 0]))
        if not _close(O[0, h], v[4, 0], 0.0):
            fails.append("single-slot O")
        if not _close(L[0, h], s, 1e-12):
            fails.append("single-slot LSE")
    return fails


def check_identical_keys(fn):
    """n slots with the same key: O = mean of their V rows, LSE = s + ln n."""
    rng = _rng(13)
    D, n = 8, 5
    q = rng.standard_normal((1, 1, D))
    key = rng.standard_normal(D)
    k = np.tile(key, (n + 2, 1, 1)).reshape(n + 2, 1, D)
    k[n] = rng.standard_normal((1, D)) * 50.0           # unselected decoys
    k[n + 1] = rng.standard_normal((1, D)) * 50.0
    v = rng.standard_normal((n + 2, 1, D))
    idx = np.array([list(range(n)) + [-1, -1]], dtype=np.int32)
    scale = 0.3
    O, L = fn(q, k, v, idx, None, scale)
    s = scale * float(q[0, 0] @ key)
    fails = []
    if not _close(O[0, 0], v[:n, 0].mean(axis=0), 1e-12):
        fails.append("identical-keys O")
    if not _close(L[0, 0], s + math.log(n), 1e-12):
        fails.append("identical-keys LSE")
    return fails


def check_duplicate_slot(fn):
    """A slot listed twice is weighted twice: (a, a, b) == (a, c, b) with slot c a copy of a."""
    rng = _rng(14)
    D = 8
    q = rng.standard_normal((1, 2, D))
    k = rng.standard_normal((4, 1, D))
    v = rng.standard_normal((4, 1, D))
    k[3], v[3] = k[0], v[0]
    scale = 0.6
    O1, L1 = fn(q, k, v, np.array([[0, 0, 1]], dtype=np.int32), None, scale)
    O2, L2 = fn(q, k, v, np.array([[0, 3, 1]], dtype=np.int32), None, scale)
    fails = []
    if not (_close(O1, O2, 1e-12) and _close(L1, L2, 1e-12)):
        fails.append("duplicate slot not weighted twice")
    s = scale * (q[0] @ k[[0, 0, 1], 0].T)             # [2, 3]
    if not _close(L1[0], logsumexp(s, axis=1), 1e-12):
        fails.append("duplicate-slot LSE vs scipy logsumexp")
    return fails


def check_invariances(fn):
    """Slot permutation, inserted padding, topk_len truncation and the slot-count filter."""
    rng = _rng(15)
    S, Hq, Hkv, D, R, K = 50, 4, 2, 8, 6, 10
    q = rng.standard_normal((R, Hq, D))
    k = rng.standard_normal((S, Hkv, D))
    v = rng.standard_normal((S, Hkv, D))
    idx = np.stack([rng.choice(S, size=K, replace=False) for _ in range(R)]).astype(np.int32)
    base_O, base_L = fn(q, k, v, idx, None, 0.25)
    fails = []
    perm = idx[:, rng.permutation(K)]
    O, L = fn(q, k, v, perm, None, 0.25)
    if not (_close(O, base_O, 1e-12) and _close(L, base_L, 1e-12)):
        fails.append("slot permutation changes the result")
    padded = np.full((R, 2 * K), -1, dtype=np.int32)
    for r in range(R):
        pos = np.sort(rng.choice(2 * K, size=K, replace=False))
        padded[r, pos] = idx[r]
    O, L = fn(q, k, v, padded, None, 0.25)
    if not (_close(O, base_O, 1e-12) and _close(L, base_L, 1e-12)):
        fails.append("-1 insertion changes the result")
    neg = padded.copy()
    neg[neg == -1] = -7
    O, L = fn(q, k, v, neg, None, 0.25)
    if not (_close(O, base_O, 1e-12) and _close(L, base_L, 1e-12)):
        fails.append("negative indices other than -1 are not padding")
    tl = rng.integers(0, K + 1, size=R).astype(np.int32)
    junk = np.concatenate([idx, rng.integers(0, S, size=(R, 3)).astype(np.int32)], axis=1)
    cut = idx.copy()
    for r in range(R):
        junk[r, tl[r]:K] = rng.integers(0, S, size=K - tl[r])
        cut[r, tl[r]:] = -1
    O1, L1 = fn(q, k, v, junk, tl, 0.25)
    O2, L2 = fn(q, k, v, cut, None, 0.25)
    if not (_close(O1, O2, 1e-12) and _close(L1, L2, 1e-12)):
        fails.append("topk_len truncation differs from a -1 tail")
    big = idx.copy()
    big[:, 0] = S + 3                                     # out of range for n_kv_slots = S
    small = idx.copy()
    small[:, 0] = -1
    k2 = np.concatenate([k, rng.standard_normal((4, Hkv, D))])
    v2 = np.concatenate([v, rng.standard_normal((4, Hkv, D))])
    O1, L1 = fn(q, k2, v2, big, None, 0.25, n_kv_slots=S)
    O2, L2 = fn(q, k2, v2, small, None, 0.25)
    if not (_close(O1, O2, 1e-12) and _close(L1, L2, 1e-12)):
        fails.append("slots >= n_kv_slots are not padding")
    return fails


def check_empty_rows(fn):
    rng = _rng(16)
    q = rng.standard_normal((3, 2, 8))
    k = rng.standard_normal((5, 1, 8))
    v = rng.standard_normal((5, 1, 8))
    idx = np.array([[-1, -1, -1], [1, 2, 3], [-1, -1, -1]], dtype=np.int32)
    tl = np.array([3, 0, 2], dtype=np.int32)
    O, L = fn(q, k, v, idx, tl, 1.0)
    fails = []
    if not (np.all(O == 0.0) and np.all(np.isneginf(L))):
        fails.append("empty rows must give O = 0, LSE = -inf")
    return fails


def check_gqa_replication(fn):
    """Hkv = 2 with KV head 1 a copy of head 0 equals Hkv = 1."""
    rng = _rng(17)
    S, D, R, K = 20, 8, 4, 6
    q = rng.standard_normal((R, 6, D))
    k1 = rng.standard_normal((S, 1, D))
    v1 = rng.standard_normal((S, 1, D))
    idx = np.stack([rng.choice(S, size=K, replace=False) for _ in range(R)]).astype(np.int32)
    O1, L1 = fn(q, k1, v1, idx, None, 0.4)
    O2, L2 = fn(q, np.concatenate([k1, k1], 1), np.concatenate([v1, v1], 1), idx, None, 0.4)
    fails = []
    if not (_close(O1, O2, 1e-12) and _close(L1, L2, 1e-12)):
        fails.append("KV-head replication changes the result")
    return fails


def check_golden(fn):
    with open(os.path.join(GOLDEN, "hand_cases.json")) as f:
        cases = json.load(f)["cases"]
    fails = []
    for c in cases:
        q = np.array(c["q"], dtype=np.float64)
        k = np.array(c["k"], dtype=np.float64)
        v = np.array(c["v"], dtype=np.float64)
        idx = np.array(c["indices"], dtype=np.int32)
        tl = None if c.get("topk_len") is None else np.array(c["topk_len"], dtype=np.int32)
        O, L = fn(q, k, v, idx, tl, c["scale"])
        wantL = np.array([[(-math.inf if x is None else x) for x in row] for row in c["lse"]])
        if not _close(O, np.array(c["out"], dtype=np.float64), 1e-12):
            fails.append(f"golden {c['name']}: O")
        if not _close(L, wantL, 1e-12):
            fails.append(f"golden {c['name']}: LSE")
    return fails


ATTENTION_CHECKS = [check_dense_equivalence, check_zero_query, check_single_slot,
                    check_identical_keys, check_duplicate_slot, check_invariances,
                    check_empty_rows, check_gqa_replication, check_golden]


# ----------------------------------------------------------------------------- union

def brute_force_union(indices, topk_len, G, n_kv_slots=0):
    """The union contract with Python sets and loops only."""
    R, K = indices.shape
    groups = []
    for g0 in range(0, R, G):
        rows = list(range(g0, min(g0 + G, R)))
        sets = []
        for r in rows:
            L = K if topk_len is None else max(0, min(int(topk_len[r]), K))
            s = set()
            for j in range(L):
                x = int(indices[r, j])
                if x >= 0 and (n_kv_slots == 0 or x < n_kv_slots):
                    s.add(x)
            sets.append(s)
        lst, bits = [], []
        for t, st in enumerate(sets):
            for x in sorted(st):
                if any(x in sets[u] for u in range(t)):
                    continue
                lst.append(x)
                bits.append(sum(1 << u for u in range(len(sets)) if x in sets[u]))
        groups.append((lst, bits))
    return groups


def union_case(seed, R=23, K=16, S=40, G=4, dup=True, with_len=True):
    """Rows that overlap without being equal: a shared base selection with some slots
    swapped for slots the row does not hold, ~15 % -1 padding, optional repeats and
    topk_len.  With dup=False every row's valid slots are distinct."""
    rng = _rng(seed)
    base = rng.choice(S, size=K, replace=False)
    idx = np.empty((R, K), dtype=np.int32)
    for r in range(R):
        row = base.copy()
        n_sw = int(rng.integers(0, K // 2))
        fresh = rng.choice(np.setdiff1d(np.arange(S), row), size=n_sw, replace=False)
        row[rng.choice(K, size=n_sw, replace=False)] = fresh
        row[rng.random(K) < 0.15] = -1
        if dup and r % 5 == 0:
            row[1] = row[0]
        idx[r] = rng.permutation(row)
    tl = rng.integers(0, K + 1, size=R).astype(np.int32) if with_len else None
    return idx, tl


def check_union_bruteforce(build):
    fails = []
    for seed, G in enumerate([2, 4, 8, 3, 1]):
        for with_len in (False, True):
            idx, tl = union_case(100 + seed, G=G, with_len=with_len)
            uidx, ubits, ulen = build(idx, tl, G)
            want = brute_force_union(idx, tl, G)
            if len(ulen) != len(want):
                fails.append(f"G={G}: group count")
                continue
            for gi, (lst, bits) in enumerate(want):
                n = int(ulen[gi])
                if n != len(lst) or list(uidx[gi, :n]) != lst or list(ubits[gi, :n]) != bits:
                    fails.append(f"G={G} group {gi}: list/bits differ from brute force")
                    break
                if np.any(uidx[gi, n:] != -1) or np.any(ubits[gi, n:] != 0):
                    fails.append(f"G={G} group {gi}: padding")
                    break
    return fails


def check_union_attention(build, attend_union, per_token):
    """Union attention with ownership bits equals per-token attention (rows without repeats)."""
    rng = _rng(200)
    R, K, S, D, Hq, Hkv = 21, 12, 35, 8, 4, 2
    idx, tl = union_case(201, R=R, K=K, S=S, G=4, dup=False)
    q = rng.standard_normal((R, Hq, D))
    k = rng.standard_normal((S, Hkv, D))
    v = rng.standard_normal((S, Hkv, D))
    fails = []
    for G in (2, 4, 8):
        uidx, ubits, ulen = build(idx, tl, G)
        O1, L1 = attend_union(q, k, v, uidx, ubits, ulen, G, 0.5)
        O2, L2 = per_token(q, k, v, idx, tl, 0.5)
        if not (_close(O1, O2, 1e-12) and _close(L1, L2, 1e-12)):
            fails.append(f"union attention != per-token (G={G})")
    return fails


# ----------------------------------------------------------------------------- paged

def paged_case(seed, with_kv_lens=True, bad_page=False):
    """Requests with contiguous per-request K/V, scattered page by page into a shuffled paged
    cache by slicing (no per-position arithmetic).  Returns the paged call's arguments and the
    per-request contiguous arrays that give the expected result."""
    rng = _rng(seed)
    ps, Hq, Hkv, D, K = 8, 4, 2, 8, 24
    rows_per_req = [3, 0, 4, 2]                 # request 1 is empty: cu_seqlens repeats
    full_pages = [5, 1, 7, 2]                   # pages holding data
    kv_lens = [37, 5, 50, 16]                   # <= full_pages * ps
    pages_per_req = max(full_pages) + 1         # trailing columns of the table are -1
    spare = 3                                   # physical pages after the mapped ones, junk
    mapped = sum(full_pages)
    perm = rng.permutation(mapped)
    kc = np.zeros(((mapped + spare) * ps, Hkv, D))
    vc = np.zeros(((mapped + spare) * ps, Hkv, D))
    kc[:] = rng.standard_normal(kc.shape)       # spare pages hold junk
    vc[:] = rng.standard_normal(vc.shape)
    table = np.full((len(full_pages), pages_per_req), -1, dtype=np.int64)
    contig_k, contig_v, off = [], [], 0
    for i, m in enumerate(full_pages):
        ki = rng.standard_normal((m * ps, Hkv, D))
        vi = rng.standard_normal((m * ps, Hkv, D))
        for pg in range(m):
            pid = int(perm[off + pg])
            table[i, pg] = pid
            kc[pid * ps:(pid + 1) * ps] = ki[pg * ps:(pg + 1) * ps]
            vc[pid * ps:(pid + 1) * ps] = vi[pg * ps:(pg + 1) * ps]
        off += m
        contig_k.append(ki)
        contig_v.append(vi)
    R = sum(rows_per_req)
    cu = np.concatenate([[0], np.cumsum(rows_per_req)]).astype(np.int64)
    q = rng.standard_normal((R, Hq, D))
    idx = np.full((R, K), -1, dtype=np.int64)
    req_rows = []
    r = 0
    for i, n in enumerate(rows_per_req):
        for _ in range(n):
            hi = pages_per_req * ps + 3           # some positions past every limit
            idx[r] = rng.integers(-2, hi, size=K)
            req_rows.append(i)
            r += 1
    tl = rng.integers(K // 2, K + 1, size=R)
    # The call declares only the mapped pages (n_pages = mapped); a table entry naming a spare
    # page (present in memory, holding junk) is then out of range and its positions are padding.
    n_pages = mapped + spare
    if bad_page:
        n_pages = mapped
        table[2, 3] = mapped + 1
    return dict(q=q, kc=kc, vc=vc, idx=idx, tl=tl, cu=cu,
                kv_lens=np.array(kv_lens) if with_kv_lens else None, table=table, ps=ps,
                n_pages=n_pages, contig_k=contig_k, contig_v=contig_v, req_rows=req_rows,
                full_pages=full_pages, kv_lens_list=kv_lens, bad_page=bad_page)


def paged_expected(c, scale):
    """Per row: the plain oracle over the request's contiguous K/V with logical positions as
    slots and the request's valid length as the slot count."""
    from oracle import sparse_prefill_rows
    R, Hq, D = c["q"].shape
    O = np.zeros((R, Hq, D))
    L = np.full((R, Hq), -np.inf)
    for r, i in enumerate(c["req_rows"]):
        n_valid = c["kv_lens_list"][i] if c["kv_lens"] is not None else c["full_pages"][i] * c["ps"]
        row = c["idx"][r].copy()
        if c["bad_page"] and i == 2:
            row[(row >= 0) & (row // c["ps"] == 3)] = -1
        Or, Lr = sparse_prefill_rows(c["q"][r:r + 1], c["contig_k"][i], c["contig_v"][i],
                                     row[None, :], c["tl"][r:r + 1], scale, [0], n_valid)
        O[r], L[r] = Or[0], Lr[0]
    return O, L


def check_paged_vs_contiguous(fn):
    fails = []
    for seed, (kvl, bad) in enumerate([(True, False), (False, False), (True, True)]):
        c = paged_case(300 + seed, with_kv_lens=kvl, bad_page=bad)
        try:
            O, L = fn(c["q"], c["kc"], c["vc"], c["idx"], c["tl"], c["cu"], c["kv_lens"],
                      c["table"], c["ps"], 0.41, c["n_pages"])
        except Exception as e:          # a translation that leaves the cache fails the pin
            fails.append(f"paged call raised {type(e).__name__} (kv_lens={kvl}, bad page={bad})")
            continue
        Oe, Le = paged_expected(c, 0.41)
        if not (_close(O, Oe, 1e-12) and _close(L, Le, 1e-12)):
            fails.append(f"paged != contiguous per request (kv_lens={kvl}, bad page={bad})")
    return fails


def check_paged_identity(fn):
    """page_size 1, one request, identity table: the indices are the physical slots."""
    from oracle import sparse_prefill
    rng = _rng(310)
    S, R, Hq, Hkv, D, K = 30, 7, 4, 1, 8, 12
    q = rng.standard_normal((R, Hq, D))
    k = rng.standard_normal((S, Hkv, D))
    v = rng.standard_normal((S, Hkv, D))
    idx = rng.integers(-1, S, size=(R, K))
    O, L = fn(q, k, v, idx, None, np.array([0, R]), None, np.arange(S)[None, :], 1, 0.3, 0)
    Oe, Le = sparse_prefill(q, k, v, idx, None, 0.3)
    return [] if (_close(O, Oe, 1e-12) and _close(L, Le, 1e-12)) else ["identity paging"]


PAGED_CHECKS = [check_paged_vs_contiguous, check_paged_identity]


# ----------------------------------------------------------------------------- MLA

def mla_case(seed, S=40, R=14, H=4, Dqk=12, Dv=8):
    """Rows at positions S-R..S-1 selecting their whole causal prefix (shuffled, -1 padded)."""
    rng = _rng(seed)
    pos = np.arange(S - R, S)
    q = rng.standard_normal((R, H, Dqk))
    kv = rng.standard_normal((S, Dqk))
    topk = S + 5
    idx = np.full((R, topk), -1, dtype=np.int64)
    for r, p in enumerate(pos):
        perm = rng.permutation(p + 1)
        slots = rng.choice(topk, size=p + 1, replace=False)
        idx[r, slots] = perm
    return q, kv, idx, pos, Dv


def check_mla_dense(fn):
    """Whole-prefix selection equals dense causal attention with keys = the full latent row and
    values = its first d_v dims (torch's math attention; LSE by scipy's logsumexp)."""
    fails = []
    for seed, (H, Dqk, Dv) in enumerate([(4, 12, 8), (1, 9, 9), (3, 16, 5)]):
        q, kv, idx, pos, Dv = mla_case(400 + seed, H=H, Dqk=Dqk, Dv=Dv)
        scale = 0.29
        O, L = fn(q, kv, idx, None, scale, Dv)
        tq = torch.from_numpy(q).permute(1, 0, 2)[None]                      # [1, H, R, Dqk]
        tk = torch.from_numpy(kv)[None, None].expand(1, H, -1, -1)
        tv = torch.from_numpy(kv[:, :Dv])[None, None].expand(1, H, -1, -1)
        keypos = torch.arange(kv.shape[0])[None, :]
        mask = torch.where(keypos <= torch.from_numpy(pos)[:, None], 0.0, float("-inf")).double()
        out = torch.ops.aten._scaled_dot_product_attention_math(tq, tk, tv, attn_mask=mask,
                                                                scale=scale)[0]
        # LSE from scipy over the masked logits (numpy float64): torch.logsumexp here was seen to
        # miss the float64 value by ~6e-10 in some runs of the suite, which is above this pin's
        # 1e-10 bound and not an error of the oracle.
        logits = scale * np.einsum("rhd,sd->hrs", q, kv)
        logits = np.where(np.arange(kv.shape[0])[None, None, :] <= pos[None, :, None], logits, -np.inf)
        Od = out[0].permute(1, 0, 2).numpy()
        Ld = logsumexp(logits, axis=-1).T
        if not (_close(O, Od, 1e-10) and _close(L, Ld, 1e-10)):
            fails.append(f"MLA dense mismatch (H={H}, d_qk={Dqk}, d_v={Dv})")
    return fails


def check_mla_vs_padded_gqa(fn):
    """The MLA layout as one KV head: key = the latent row, value = its first d_v dims padded
    with zeros to d_qk.  The plain (pinned) oracle must give O in the first d_v dims, zeros
    after, and the same LSE; topk_len and padding included."""
    from oracle import sparse_prefill
    rng = _rng(410)
    R, S, H, Dqk, Dv, K = 9, 30, 5, 12, 7, 20
    q = rng.standard_normal((R, H, Dqk))
    kv = rng.standard_normal((S, Dqk))
    idx = rng.integers(-2, S, size=(R, K))
    tl = rng.integers(0, K + 1, size=R)
    tl[0] = 0                                   # rows with no valid slot: O = 0, LSE = -inf
    idx[1] = -1
    O, L = fn(q, kv, idx, tl, 0.37, Dv)
    vpad = np.concatenate([kv[:, :Dv], np.zeros((S, Dqk - Dv))], axis=1)
    Og, Lg = sparse_prefill(q, kv[:, None, :], vpad[:, None, :], idx, tl, 0.37)
    ok = _close(O, Og[:, :, :Dv], 1e-12) and _close(L, Lg, 1e-12) and np.all(Og[:, :, Dv:] == 0)
    return [] if ok else ["MLA != padded single-KV-head attention"]


MLA_CHECKS = [check_mla_dense, check_mla_vs_padded_gqa]


# ----------------------------------------------------------------------------- page split

def page_pool_case(seed, n_pages=6, src_ps=8, sections=(32, 16, 48)):
    """A source pool built from per-(page, token, section) byte blocks with array reshapes, and
    the expected destination for each split ratio built the same way (no per-token offsets)."""
    rng = _rng(seed)
    blocks = [rng.integers(0, 256, size=(n_pages, src_ps, sb), dtype=np.uint8) for sb in sections]
    # page p = concatenation over sections of blocks[k][p] flattened (token-major)
    src = np.concatenate([np.concatenate([b[p].reshape(-1) for b in blocks]) for p in range(n_pages)])

    def expected(dst_ps):
        ratio = src_ps // dst_ps
        pages = []
        for p in range(n_pages):
            for i in range(ratio):
                pages.append(np.concatenate([b[p, i * dst_ps:(i + 1) * dst_ps].reshape(-1)
                                             for b in blocks]))
        return np.concatenate(pages)
    return src, expected, list(sections)


def check_page_split(split):
    """split(src, dst, n_pages, src_ps, dst_ps, sections, mark) -> new dst (flat uint8)."""
    fails = []
    src, expected, secs = page_pool_case(500)
    for dst_ps in (8, 4, 2, 1):
        got = split(src, np.zeros_like(src), 6, 8, dst_ps, secs, None)
        if not np.array_equal(got, expected(dst_ps)):
            fails.append(f"full split to pages of {dst_ps}")
    # masked: touched pages equal the full split, the others keep their stale bytes
    stale = _rng(501).integers(0, 256, size=src.size, dtype=np.uint8)
    mark = np.array([0, 1, 0, 0, 1, 1], dtype=np.uint8)
    got = split(src, stale, 6, 8, 2, secs, mark)
    full = expected(2)
    pb = 8 * sum(secs)                         # page bytes are the same for both page sizes x ratio
    for p in range(6):
        want = full[p * pb:(p + 1) * pb] if mark[p] else stale[p * pb:(p + 1) * pb]
        if not np.array_equal(got[p * pb:(p + 1) * pb], want):
            fails.append(f"masked split, source page {p} (marked={bool(mark[p])})")
    return fails


def check_page_mark(mark_fn):
    """mark_fn(indices, src_ps, n_pages) -> uint8 [n_pages]; against the set of pages of the
    valid indices (padding and slots past the pool ignored)."""
    rng = _rng(510)
    idx = rng.integers(-3, 9 * 16 + 20, size=(5, 23))
    got = mark_fn(idx, 16, 9)
    want = np.zeros(9, dtype=np.uint8)
    for page in {int(t) // 16 for t in idx.reshape(-1) if 0 <= t < 9 * 16}:
        want[page] = 1
    fails = [] if np.array_equal(got, want) else ["page mark != set of touched pages"]
    # hand-chosen page boundaries: 15 -> page 0, 16 -> 1, 47 -> 2, 100 -> 6, 143 -> 8, 200 past
    got = mark_fn(np.array([[15, 16, -1, 47], [100, 143, -2, 200]]), 16, 9)
    if not np.array_equal(got, np.array([1, 1, 1, 0, 0, 0, 1, 0, 1], dtype=np.uint8)):
        fails.append("page boundaries")
    if mark_fn(np.full((2, 3), -1), 16, 9).any():
        fails.append("padding marked a page")
    return fails


# ----------------------------------------------------------------------------- FP8 KV cache

def check_e4m3_decode(decode):
    """Every code against torch's float8_e4m3fn conversion, plus hand-checked values."""
    codes = np.arange(256, dtype=np.uint8)
    got = decode(codes)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    fails = []
    if not np.array_equal(np.isnan(got), np.isnan(want)) or \
            not np.array_equal(got[~np.isnan(got)], want[~np.isnan(want)]):
        fails.append("e4m3 decode != torch float8_e4m3fn")
    hand = {0x38: 1.0, 0x7E: 448.0, 0xFE: -448.0, 0x01: 2.0 ** -9, 0x08: 2.0 ** -6,
            0x3C: 1.5, 0x40: 2.0, 0x30: 0.5}
    for c, v in hand.items():
        if decode(np.array([c], dtype=np.uint8))[0] != v:
            fails.append(f"code 0x{c:02x}")
    if not (np.signbit(decode(np.array([0x80], dtype=np.uint8))[0]) and
            decode(np.array([0x80], dtype=np.uint8))[0] == 0.0):
        fails.append("code 0x80 is -0")
    return fails


def check_fp8_attention(fn):
    """fn(q, k8, v8, k_scale, v_scale, page_size, idx, tl, scale) equals the plain (pinned)
    oracle on caches the test dequantises with torch (float8 -> float64, times the page scale
    broadcast over each page's slots)."""
    from oracle import sparse_prefill
    rng = _rng(600)
    R, S, Hq, Hkv, D, K, ps = 7, 40, 4, 2, 16, 25, 8
    q = rng.standard_normal((R, Hq, D))
    k8 = rng.integers(0, 256, size=(S, Hkv, D), dtype=np.uint8)
    v8 = rng.integers(0, 256, size=(S, Hkv, D), dtype=np.uint8)
    k8[(k8 & 0x7F) == 0x7F] = 0x11                # keep NaN codes out of the attention check
    v8[(v8 & 0x7F) == 0x7F] = 0x22
    ksc = rng.uniform(0.01, 0.2, size=(S // ps, Hkv))
    vsc = rng.uniform(0.5, 3.0, size=(S // ps, Hkv))
    idx = rng.integers(-1, S, size=(R, K))
    tl = rng.integers(0, K + 1, size=R)

    def deq(c, sc):
        vals = torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64)
        per_slot = torch.from_numpy(sc).repeat_interleave(ps, dim=0)            # [S, Hkv]
        return (vals * per_slot[:, :, None]).numpy()
    O, L = fn(q, k8, v8, ksc, vsc, ps, idx, tl, 0.3)
    Oe, Le = sparse_prefill(q, deq(k8, ksc), deq(v8, vsc), idx, tl, 0.3)
    return [] if (_close(O, Oe, 1e-12) and _close(L, Le, 1e-12)) else ["FP8 attention != dequantised"]
