"""The MLA-shaped kernel (qsa_sparse_mla_prefill: d_qk 576, d_v 512, one latent KV row per slot)
against the MLA oracle, per-token and union, small cases in full and the 8192-token workloads on
sampled rows (GPU only).  Bounds: O max-abs 2e-2, LSE relative 1e-3 (helpers.py)."""
import numpy as np
import pytest

import oracle
from helpers import assert_parity
from top_sparse_attention_row_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from top_sparse_attention_row_gb300 import build, binding
    build.build()
    binding.load_library()
    return binding


def dev(w):
    import torch
    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()
    q = bf(w.q)
    kv = bf(w.k.reshape(w.k.shape[0], -1))
    idx = torch.from_numpy(np.ascontiguousarray(w.indices, dtype=np.int32)).cuda()
    tl = None if w.topk_len is None else torch.from_numpy(np.ascontiguousarray(w.topk_len, dtype=np.int32)).cuda()
    return q, kv, idx, tl


def run(B, w, union_g=0, n_kv_slots=0):
    import torch
    q, kv, idx, tl = dev(w)
    out, lse = B.sparse_mla_prefill(q, kv, idx, tl, w.scale, union_g=union_g, n_kv_slots=n_kv_slots)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    return out, lse


def ref(w, rows=None, n_kv_slots=0):
    rows = np.arange(w.n_rows) if rows is None else rows
    return oracle.sparse_mla_prefill_rows(w.q, w.k.reshape(w.k.shape[0], -1), w.indices, w.topk_len,
                                          w.scale, rows, 512, n_kv_slots)


def chunk_mla(n_rows, context, n_heads, topk, seed):
    """n_rows rows at the end of a context, uniform causal selections (several tiles + tail)."""
    rng = np.random.default_rng(seed)
    pos = np.arange(context - n_rows, context)
    q = W.randn_bf16(rng, (n_rows, n_heads, 576))
    kv = W.randn_bf16(rng, (context, 1, 576))
    idx = W.causal_uniform_indices(rng, pos, topk)
    return W.Workload("mla_chunk", q, kv, kv[:, :, :512], idx, None, 1.0 / 24.0, pos)


@pytest.mark.parametrize("heads", [8, 1, 16, 32, 40])
def test_mla_multi_tile_ragged(B, heads):
    # 2051 slots = 16 full tiles + a 3-slot tail; early rows have short prefixes
    w = chunk_mla(n_rows=48, context=2300, n_heads=heads, topk=2051, seed=heads)
    out, lse = run(B, w)
    O, L = ref(w)
    assert_parity(out, lse, O, L, what=f"mla {heads} heads")


@pytest.mark.parametrize("topk", [1, 17, 128, 129, 640])
def test_mla_topk_widths(B, topk):
    w = chunk_mla(n_rows=40, context=900, n_heads=8, topk=topk, seed=100 + topk)
    out, lse = run(B, w)
    O, L = ref(w)
    assert_parity(out, lse, O, L, what=f"mla topk {topk}")


@pytest.mark.parametrize("G,heads", [(2, 8), (4, 8), (2, 16), (3, 8)])
def test_mla_union_equals_per_token_oracle(B, G, heads):
    w = W.make_mla(seed=20 + G, n_rows=601, topk=256, n_heads=heads, name="mla_union_small")
    before = B.counters()
    out, lse = run(B, w, union_g=G)
    after = B.counters()
    assert after["calls_union"] == before["calls_union"] + 1
    O, L = ref(w)
    assert_parity(out, lse, O, L, what=f"mla union G={G} heads={heads}")


def test_mla_union_fallback_counted(B):
    w = W.make_mla(seed=30, n_rows=64, topk=128, n_heads=16, name="mla_fallback")
    before = B.counters()
    out, lse = run(B, w, union_g=4)                      # 4 x 16 = 64 columns > 32
    after = B.counters()
    assert after["union_fallbacks"] == before["union_fallbacks"] + 1
    O, L = ref(w)
    assert_parity(out, lse, O, L, what="mla union fallback")


def test_mla_edge_rows(B):
    """All -1, topk_len 0 and short, other negatives, duplicates (weighted twice), slots past
    n_kv_slots."""
    w = chunk_mla(n_rows=10, context=700, n_heads=8, topk=300, seed=55)
    idx = w.indices.copy()
    tl = np.full(10, 300, dtype=np.int32)
    idx[0] = -1
    tl[1] = 0
    tl[2] = 5
    idx[3, ::4] = -7
    idx[4, 10:20] = idx[4, 0:10]                           # duplicates
    idx[5, 0:30] = 650                                     # >= n_kv_slots below: padding
    w = W.Workload("mla_edge", w.q, w.k, w.v, idx, tl, w.scale, w.positions)
    out, lse = run(B, w, n_kv_slots=600)
    O, L = ref(w, n_kv_slots=600)
    assert np.isneginf(L[0]).all() and np.isneginf(L[1]).all()
    assert_parity(out, lse, O, L, what="mla edge rows")


@pytest.mark.parametrize("G", [0, 2, 4])
def test_mla_full_size_8k(B, oracle_pool, G):
    """The 8192-token MLA prefill (8 heads, topk 2048, random walk) as the benchmark runs it,
    every row against the oracle."""
    w = W.make("mla_8k")
    out, lse = run(B, w, union_g=G)
    oracle_pool.check_all_rows(("mla_8k", ""), "mla", out, lse, f"mla_8k G={G}")


def paged_mla_case(seed=70, ps=64, kv_lens=(700, 1300, 400), rows=(30, 50, 20), topk=512, heads=8):
    """Three requests whose latent rows live on shuffled pages of one cache (two spare pages),
    rows at the end of each request selecting distinct causal positions of it; returns the
    paged call's inputs."""
    rng = np.random.default_rng(seed)
    pages = [-(-L // ps) for L in kv_lens]
    n_pages = sum(pages) + 2
    perm = rng.permutation(n_pages)
    cache = W.randn_bf16(rng, (n_pages * ps, 576))
    table = np.full((len(kv_lens), max(pages) + 1), -1, dtype=np.int32)
    off = 0
    for i, n in enumerate(pages):
        table[i, :n] = perm[off:off + n]
        off += n
    R = sum(rows)
    q = W.randn_bf16(rng, (R, heads, 576))
    logical = np.full((R, topk), -1, dtype=np.int32)
    cu = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    r = 0
    for i, (L, n) in enumerate(zip(kv_lens, rows)):
        for pos in range(L - n, L):
            m = min(pos + 1, topk)
            logical[r, :m] = rng.choice(pos + 1, size=m, replace=False)
            r += 1
    return q, cache, logical, cu, np.asarray(kv_lens, dtype=np.int32), table, ps, n_pages


@pytest.mark.parametrize("G", [0, 2])
def test_mla_paged_matches_oracle_and_plain_entry(B, G):
    import torch
    q, cache, logical, cu, kvl, table, ps, n_pages = paged_mla_case()
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    dq, dkv = bf(q), bf(cache)
    out, lse = B.sparse_mla_prefill_paged(dq, dkv, i32(logical), None, i32(cu), i32(kvl), i32(table),
                                          ps, 1.0 / 24.0, n_pages=n_pages, union_g=G)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    phys = oracle.physical_indices(logical, cu, kvl, table, ps, n_pages)
    O, L = oracle.sparse_mla_prefill(q, cache, phys, None, 1.0 / 24.0)
    assert_parity(out, lse, O, L, what=f"mla paged G={G}")
    out2, lse2 = B.sparse_mla_prefill(dq, dkv, i32(np.where(phys >= 0, phys, -1)), None, 1.0 / 24.0,
                                      union_g=G)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse, lse2)
