"""Seeded synthetic workloads for top-k sparse attention prefill.

This module only draws inputs: bf16 query / key / value tensors, top-k index
rows, per-row ``topk_len`` and (for the paged case) a shuffled page table.  It
holds none of the attention arithmetic, so the CPU oracle and the CUDA path
can both be fed from it without sharing any of the method's code.

Everything is numpy, seeded through ``numpy.random.default_rng``.  bf16
tensors are returned as raw ``uint16`` bit patterns (round-to-nearest-even
from float32 draws of N(0, 1)); ``bf16_to_f32`` widens them exactly.

Workload shapes follow the pages' benchmarks:

* "[QSA] Tune sm120 sparse prefill geometry", Kernel measurements: batch 1,
  chunk of 8192 query rows at the end of a 32k / 128k context, 2051 selected
  slots per row, head_dim 256, group 6 (6 Q / 1 KV) and group 12 (12 Q / 1 KV,
  24 Q / 2 KV).
* "DSA prefill ... triton_sparse_mla", Modifications (union table) and the
  measurement note on the calibrated random walk: token t+1 repeats token t's
  selection with about 2 % of its entries swapped, and tokens t < topk select
  their whole visible prefix with -1 padding.
* A chunked mixed batch over a paged cache (page size 64, shuffled page
  table); indices are physical slots, with per-row ``topk_len``.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

HEAD_DIM = 256


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest-even) and return the bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def randn_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


@dataclass
class Workload:
    """One sparse-prefill problem.

    q: [n_rows, n_qheads, D] bf16 bits; k, v: [n_slots, n_kvheads, D] bf16 bits;
    indices: [n_rows, topk] int32 physical slots, -1 = padding;
    topk_len: [n_rows] int32 or None (None = every slot of the row is considered).
    """
    name: str
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    indices: np.ndarray
    topk_len: Optional[np.ndarray]
    scale: float
    positions: np.ndarray                      # absolute causal position of each row
    meta: dict = field(default_factory=dict)

    @property
    def n_rows(self) -> int:
        return int(self.q.shape[0])

    @property
    def n_qheads(self) -> int:
        return int(self.q.shape[1])

    @property
    def n_kvheads(self) -> int:
        return int(self.k.shape[1])

    @property
    def n_slots(self) -> int:
        return int(self.k.shape[0])

    @property
    def head_dim(self) -> int:
        return int(self.q.shape[2])

    @property
    def topk(self) -> int:
        return int(self.indices.shape[1])

    def valid_counts(self) -> np.ndarray:
        """Number of considered, non-negative slots per row (the v_r of the roofline)."""
        idx = self.indices
        mask = idx >= 0
        if self.topk_len is not None:
            cols = np.arange(idx.shape[1])[None, :]
            mask &= cols < np.clip(self.topk_len, 0, idx.shape[1])[:, None]
        return mask.sum(axis=1)


def causal_uniform_indices(rng: np.random.Generator, positions: np.ndarray, topk: int) -> np.ndarray:
    """Row at position p: min(p+1, topk) distinct positions drawn uniformly from [0, p],
    stored in random slot order, -1 in the remaining slots."""
    out = np.full((len(positions), topk), -1, dtype=np.int32)
    for r, p in enumerate(positions):
        n = min(int(p) + 1, topk)
        out[r, :n] = rng.choice(int(p) + 1, size=n, replace=False)
    return out


def random_walk_indices(rng: np.random.Generator, n_rows: int, topk: int,
                        swap_frac: float = 0.02) -> np.ndarray:
    """Calibrated random walk for a prefill from position 0.

    Token t < topk selects all of [0, t] (shuffled), -1 after.  Token t >= topk
    repeats token t-1's row with m = min(round(swap_frac*topk), t+1-topk) of its
    slots replaced by fresh positions from [0, t] that the row does not hold.
    """
    n_swap = max(1, int(round(swap_frac * topk)))
    out = np.full((n_rows, topk), -1, dtype=np.int32)
    member = np.zeros(n_rows, dtype=bool)
    row = None
    for t in range(n_rows):
        if t < topk:
            out[t, : t + 1] = rng.permutation(t + 1)
            if t == topk - 1:
                row = out[t].copy()
                member[row] = True
            continue
        avail = np.flatnonzero(~member[: t + 1])
        m = min(n_swap, len(avail))
        slots = rng.choice(topk, size=m, replace=False)
        fresh = rng.choice(avail, size=m, replace=False)
        member[row[slots]] = False
        row[slots] = fresh
        member[fresh] = True
        out[t] = row
    return out


def make_tiny(seed: int = 0) -> Workload:
    """Batch 1, context 512, 256 query rows at positions 256..511, 6 Q / 1 KV, topk 128."""
    rng = np.random.default_rng(seed)
    S, R, Hq, Hkv, K = 512, 256, 6, 1, 128
    pos = np.arange(S - R, S)
    q = randn_bf16(rng, (R, Hq, HEAD_DIM))
    k = randn_bf16(rng, (S, Hkv, HEAD_DIM))
    v = randn_bf16(rng, (S, Hkv, HEAD_DIM))
    idx = causal_uniform_indices(rng, pos, K)
    return Workload("tiny", q, k, v, idx, None, 1.0 / 16.0, pos)


def make_chunk(n_rows: int, context: int, n_qheads: int, n_kvheads: int, topk: int,
               seed: int, name: str) -> Workload:
    """A chunk of ``n_rows`` query rows at the end of a ``context``-token prefix-cached
    prompt; every row draws uniformly from its causal prefix."""
    rng = np.random.default_rng(seed)
    pos = np.arange(context - n_rows, context)
    q = randn_bf16(rng, (n_rows, n_qheads, HEAD_DIM))
    k = randn_bf16(rng, (context, n_kvheads, HEAD_DIM))
    v = randn_bf16(rng, (context, n_kvheads, HEAD_DIM))
    idx = causal_uniform_indices(rng, pos, topk)
    return Workload(name, q, k, v, idx, None, 1.0 / 16.0, pos)


def make_group6(seed: int = 1, n_rows: int = 8192, context: int = 32768) -> Workload:
    """Group 6: 8192 rows at the end of a 32768 context, 6 Q / 1 KV, topk 2051."""
    return make_chunk(n_rows, context, 6, 1, 2051, seed, "group6_32k")


def make_group12(seed: int = 2, n_rows: int = 8192, context: int = 131072,
                 n_qheads: int = 24, n_kvheads: int = 2) -> Workload:
    """Group 12: 8192 rows at the end of a 131072 context, topk 2051 (24 Q / 2 KV by default,
    12 Q / 1 KV as the alternative rank shape)."""
    return make_chunk(n_rows, context, n_qheads, n_kvheads, 2051, seed,
                      f"group12_128k_{n_qheads}q{n_kvheads}kv")


def make_rows(n_rows: int, seed: int = 9) -> Workload:
    """Query-count sweep point: ``n_rows`` rows at the end of an 8192-token context (the rest a
    prefix), group 6, topk 2051, so each row gathers all 2051 of its slots ("[QSA] Tune sm120 sparse
    prefill geometry", Query-count sweep)."""
    return make_chunk(n_rows, 8192, 6, 1, 2051, seed + n_rows, f"rows{n_rows}_8k")


def make_union(seed: int = 3, n_rows: int = 8192, topk: int = 2048) -> Workload:
    """Prefill of n_rows tokens from position 0, 8 Q / 1 KV, topk 2048, random-walk indices."""
    rng = np.random.default_rng(seed)
    S = n_rows
    pos = np.arange(n_rows)
    q = randn_bf16(rng, (n_rows, 8, HEAD_DIM))
    k = randn_bf16(rng, (S, 1, HEAD_DIM))
    v = randn_bf16(rng, (S, 1, HEAD_DIM))
    idx = random_walk_indices(rng, n_rows, topk)
    return Workload("union_8k", q, k, v, idx, None, 1.0 / 16.0, pos)


def quantize_e4m3(bits: np.ndarray, page_size: int):
    """bf16 bit patterns [S, Hkv, D] -> (e4m3 codes [S, Hkv, D] uint8, fp32 scales
    [ceil(S / page_size), Hkv]): one scale per page and KV head, amax / 448, values rounded to
    the nearest e4m3 by torch's float8_e4m3fn cast (input preparation for the FP8 cache path)."""
    import torch
    x = torch.from_numpy(bf16_to_f32(bits))
    S, H, D = x.shape
    pages = -(-S // page_size)
    pad = pages * page_size - S
    xp = torch.cat([x, torch.zeros(pad, H, D)]) if pad else x
    amax = xp.reshape(pages, page_size, H, D).abs().amax(dim=(1, 3))           # [pages, H]
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax)).float()
    per_slot = scale.repeat_interleave(page_size, dim=0)[:S]                    # [S, H]
    codes = (x / per_slot[:, :, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.numpy(), scale.numpy()


def with_fp8_cache(w: Workload, page_size: int = 64) -> Workload:
    """The same workload with K and V held as an e4m3 cache with per-page scales
    (meta: k8, v8, k_scale, v_scale, page_size)."""
    k8, ks = quantize_e4m3(w.k, page_size)
    v8, vs = quantize_e4m3(w.v, page_size)
    meta = dict(w.meta, fp8=True, k8=k8, v8=v8, k_scale=ks, v_scale=vs, fp8_page_size=page_size)
    return Workload(w.name + "_fp8", w.q, w.k, w.v, w.indices, w.topk_len, w.scale, w.positions, meta)


MLA_DQK, MLA_DV = 576, 512


def make_mla(seed: int = 5, n_rows: int = 8192, topk: int = 2048, n_heads: int = 8,
             name: str = "mla_8k", indices: str = "walk") -> Workload:
    """MLA-shaped prefill of n_rows tokens from position 0: n_heads query heads of 576 dims over
    one latent KV row per token (576 dims as key, the first 512 as value), topk 2048.  Indices:
    "walk" = the calibrated random walk of the union workload, "uniform" = distinct uniform
    positions of each row's causal prefix.  k holds the latent rows as [S, 1, 576] and v is the
    view of their first 512 dims; scale = 1/sqrt(576)."""
    rng = np.random.default_rng(seed)
    pos = np.arange(n_rows)
    q = randn_bf16(rng, (n_rows, n_heads, MLA_DQK))
    kv = randn_bf16(rng, (n_rows, 1, MLA_DQK))
    if indices == "walk":
        idx = random_walk_indices(rng, n_rows, topk)
    else:
        idx = causal_uniform_indices(rng, pos, topk)
    return Workload(name, q, kv, kv[:, :, :MLA_DV], idx, None, 1.0 / 24.0, pos,
                    dict(mla=True, d_v=MLA_DV))


def make_mixed(seed: int = 4, new_tokens=(512, 2048, 4096, 8192),
               prefixes=(0, 16384, 32768, 65536), page_size: int = 64,
               n_qheads: int = 6, n_kvheads: int = 1, topk: int = 2051) -> Workload:
    """Chunked mixed batch over a paged cache.

    Request i holds prefixes[i] + new_tokens[i] logical KV positions in whole pages of
    ``page_size``; physical pages are a seeded permutation.  Row r of request i sits at
    logical position p = prefixes[i] + j and selects min(p+1, topk) distinct positions of
    [0, p], translated to physical slots page_table[i][p // page_size]*page_size + p % page_size.
    ``topk_len`` = min(p+1, topk); slots past it hold -1.
    """
    rng = np.random.default_rng(seed)
    kv_lens = [p + n for p, n in zip(prefixes, new_tokens)]
    pages_per_req = [-(-L // page_size) for L in kv_lens]
    n_pages = int(sum(pages_per_req))
    perm = rng.permutation(n_pages).astype(np.int64)
    page_tables, off = [], 0
    for n in pages_per_req:
        page_tables.append(perm[off:off + n])
        off += n
    S = n_pages * page_size
    R = int(sum(new_tokens))
    q = randn_bf16(rng, (R, n_qheads, HEAD_DIM))
    k = randn_bf16(rng, (S, n_kvheads, HEAD_DIM))
    v = randn_bf16(rng, (S, n_kvheads, HEAD_DIM))
    idx = np.full((R, topk), -1, dtype=np.int32)
    logical_idx = np.full((R, topk), -1, dtype=np.int32)
    tlen = np.zeros(R, dtype=np.int32)
    pos = np.zeros(R, dtype=np.int64)
    req_of_row = np.zeros(R, dtype=np.int32)
    r = 0
    for i, (pre, new) in enumerate(zip(prefixes, new_tokens)):
        pt = page_tables[i]
        for j in range(new):
            p = pre + j
            n = min(p + 1, topk)
            logical = rng.choice(p + 1, size=n, replace=False)
            logical_idx[r, :n] = logical
            idx[r, :n] = pt[logical // page_size] * page_size + logical % page_size
            tlen[r] = n
            pos[r] = p
            req_of_row[r] = i
            r += 1
    # The same batch as the paged call takes it: logical positions, ragged row offsets and one
    # page-table row per request (-1 past the request's pages).
    table = np.full((len(page_tables), max(pages_per_req)), -1, dtype=np.int32)
    for i, pt in enumerate(page_tables):
        table[i, :len(pt)] = pt
    cu_seqlens_q = np.concatenate([[0], np.cumsum(new_tokens)]).astype(np.int32)
    meta = dict(page_size=page_size, page_tables=page_tables, prefixes=list(prefixes),
                new_tokens=list(new_tokens), kv_lens=kv_lens, req_of_row=req_of_row,
                logical_indices=logical_idx, page_table=table, cu_seqlens_q=cu_seqlens_q,
                kv_lens_array=np.asarray(kv_lens, dtype=np.int32), n_pages=n_pages)
    return Workload("mixed_paged", q, k, v, idx, tlen, 1.0 / 16.0, pos, meta)


def make_page_split(seed: int = 8, n_src_pages: int = 4096, src_page_size: int = 256,
                    dst_page_size: int = 64, batch: int = 8, window: int = 512,
                    section_bytes=(512, 16, 128)) -> dict:
    """A decode step's page re-layout: a pool of n_src_pages pages of src_page_size tokens, each
    token 656 bytes in three sections (512 fp8 latent bytes, 16 bytes of scales, 128 bytes of
    bf16 rope), split to pages of dst_page_size.  Each of `batch` requests owns a random set of
    physical pages; its decode row selects the last `window` tokens of its context, so about
    two source pages per request are touched.  Returns the pool bytes (uint8, flat), indices
    [batch, window] int32 source slots and the shape."""
    rng = np.random.default_rng(seed)
    token_bytes = int(sum(section_bytes))
    pool = rng.integers(0, 256, size=n_src_pages * src_page_size * token_bytes, dtype=np.uint8)
    perm = rng.permutation(n_src_pages)
    pages_per_req = n_src_pages // batch
    idx = np.empty((batch, window), dtype=np.int32)
    for b in range(batch):
        pages = perm[b * pages_per_req:(b + 1) * pages_per_req]
        ctx = int(rng.integers(window, pages_per_req * src_page_size))
        logical = np.arange(ctx - window, ctx)
        idx[b] = pages[logical // src_page_size] * src_page_size + logical % src_page_size
    return dict(pool=pool, indices=idx, n_src_pages=n_src_pages, src_page_size=src_page_size,
                dst_page_size=dst_page_size, section_bytes=list(section_bytes))


CONFIGS = {
    "tiny": make_tiny,
    "group6_32k": make_group6,
    "group12_128k": make_group12,
    "group12_128k_12q1kv": lambda seed=2: make_group12(seed, n_qheads=12, n_kvheads=1),
    "union_8k": make_union,
    "mixed_paged": make_mixed,
    "mla_8k": make_mla,
    "mla_4k": lambda seed=6: make_mla(seed, n_rows=4096, name="mla_4k"),
    "mla_2k": lambda seed=7: make_mla(seed, n_rows=2048, name="mla_2k"),
}
# query-count sweep at KV 8192
for _r in (32, 64, 128, 256, 512, 1024):
    CONFIGS[f"rows{_r}_8k"] = (lambda r: (lambda seed=9: make_rows(r, seed)))(_r)


def make(name: str, **kw) -> Workload:
    return CONFIGS[name](**kw)


def union_size_ratio(indices: np.ndarray, G: int, start_row: int = 0) -> float:
    """Mean size of the union of G consecutive rows' valid sets over the mean row size
    (the calibration figure of the random-walk generator)."""
    idx = indices[start_row:]
    n_groups = idx.shape[0] // G
    uni, own = 0, 0
    for gi in range(n_groups):
        rows = idx[gi * G:(gi + 1) * G]
        sets = [set(r[r >= 0].tolist()) for r in rows]
        uni += len(set().union(*sets))
        own += sum(len(s) for s in sets) / G
    return uni / own
