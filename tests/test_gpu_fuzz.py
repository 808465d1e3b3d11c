"""Seeded random configurations of every attention entry point against the oracle (GPU only).

Each case draws its shape (rows, heads, group, top-k, union size, page size) and its index
pathologies (padding, other negatives, slots past the cache with a slot count, duplicates for
the per-token path, topk_len) from a fixed seed, so a failure names a reproducible case.
Bounds: O max-abs 2e-2, LSE relative 1e-3 (helpers.py)."""
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


def cuda(a, bf16=False):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if bf16 else np.ascontiguousarray(a))
    return (t.view(torch.bfloat16) if bf16 else t).cuda()


def random_indices(rng, R, K, S, dup, junk):
    """Distinct slots per row (plus duplicates when dup), with padding, other negatives and, when
    junk, slots past S; returns indices and topk_len (or None)."""
    idx = np.full((R, K), -1, dtype=np.int32)
    for r in range(R):
        n = int(rng.integers(0, min(K, S) + 1))
        idx[r, :n] = rng.choice(S, size=n, replace=False)
        rng.shuffle(idx[r])
    if dup and K >= 4:
        rows = rng.choice(R, size=max(1, R // 5), replace=False)
        for r in rows:
            a, b = rng.choice(K, size=2, replace=False)
            idx[r, a] = idx[r, b]
    neg = rng.random(idx.shape) < 0.03
    idx[neg] = -rng.integers(2, 50, size=int(neg.sum()))
    if junk:
        far = rng.random(idx.shape) < 0.03
        idx[far] = S + rng.integers(0, 99, size=int(far.sum()))
    tl = rng.integers(0, K + 1, size=R).astype(np.int32) if rng.random() < 0.5 else None
    return idx, tl


@pytest.mark.parametrize("case", range(24))
def test_fuzz_d256(B, case):
    import torch
    rng = np.random.default_rng(1000 + case)
    Hkv = int(rng.choice([1, 2, 3]))
    g = int(rng.integers(1, 41))
    Hq = g * Hkv
    R = int(rng.integers(1, 200))
    S = int(rng.integers(16, 1500))
    K = int(rng.integers(1, 700))
    G = int(rng.choice([0, 0, 2, 3, 4, 8]))
    q = W.randn_bf16(rng, (R, Hq, 256))
    k = W.randn_bf16(rng, (S, Hkv, 256))
    v = W.randn_bf16(rng, (S, Hkv, 256))
    idx, tl = random_indices(rng, R, K, S, dup=(G == 0), junk=True)
    out, lse = B.sparse_prefill(cuda(q, True), cuda(k, True), cuda(v, True), cuda(idx),
                                None if tl is None else cuda(tl), 1.0 / 16.0, union_g=G, n_kv_slots=S)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    O, L = oracle.sparse_prefill(q, k, v, idx, tl, 1.0 / 16.0, n_kv_slots=S)
    assert_parity(out, lse, O, L, what=f"case {case}: R={R} Hq={Hq} Hkv={Hkv} K={K} S={S} G={G}")


@pytest.mark.parametrize("case", range(10))
def test_fuzz_fp8(B, case):
    import torch
    rng = np.random.default_rng(2000 + case)
    Hkv = int(rng.choice([1, 2]))
    g = int(rng.integers(1, 33))
    Hq = g * Hkv
    R, S, K = int(rng.integers(1, 120)), int(rng.integers(16, 900)), int(rng.integers(1, 400))
    ps = int(rng.choice([1, 16, 64, 100]))
    G = int(rng.choice([0, 2, 4]))
    q = W.randn_bf16(rng, (R, Hq, 256))
    k = W.randn_bf16(rng, (S, Hkv, 256))
    v = W.randn_bf16(rng, (S, Hkv, 256))
    idx, tl = random_indices(rng, R, K, S, dup=(G == 0), junk=True)
    k8, ks = W.quantize_e4m3(k, ps)
    v8, vs = W.quantize_e4m3(v, ps)
    out, lse = B.sparse_prefill_fp8(cuda(q, True), cuda(k8), cuda(v8), cuda(ks), cuda(vs), ps,
                                    cuda(idx), None if tl is None else cuda(tl), 1.0 / 16.0,
                                    union_g=G, n_kv_slots=S)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    O, L = oracle.sparse_prefill_fp8(q, k8, v8, ks, vs, ps, idx, tl, 1.0 / 16.0, n_kv_slots=S)
    assert_parity(out, lse, O, L, what=f"fp8 case {case}: Hq={Hq} Hkv={Hkv} K={K} ps={ps} G={G}")


@pytest.mark.parametrize("case", range(10))
def test_fuzz_paged(B, case):
    import torch
    rng = np.random.default_rng(3000 + case)
    n_req = int(rng.integers(1, 7))
    ps = int(rng.choice([1, 8, 48, 64, 128]))
    Hkv, g = int(rng.choice([1, 2])), int(rng.integers(1, 17))
    Hq, K = g * Hkv, int(rng.integers(1, 300))
    kv_lens = rng.integers(1, 800, size=n_req)
    rows = rng.integers(0, 40, size=n_req)
    rows[0] = max(rows[0], 1)
    pages = -(-kv_lens // ps)
    n_pages = int(pages.sum()) + 3
    perm = rng.permutation(n_pages)
    table = np.full((n_req, int(pages.max()) + 1), -1, dtype=np.int32)
    off = 0
    for i in range(n_req):
        table[i, :pages[i]] = perm[off:off + pages[i]]
        off += pages[i]
    R = int(rows.sum())
    cu = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    logical = np.full((R, K), -1, dtype=np.int32)
    r = 0
    for i in range(n_req):
        for _ in range(rows[i]):
            n = int(rng.integers(0, min(K, kv_lens[i]) + 1))
            logical[r, :n] = rng.choice(int(kv_lens[i]) + 5, size=n, replace=False)   # some past kv_len
            r += 1
    S = n_pages * ps
    q = W.randn_bf16(rng, (R, Hq, 256))
    k = W.randn_bf16(rng, (S, Hkv, 256))
    v = W.randn_bf16(rng, (S, Hkv, 256))
    G = int(rng.choice([0, 2, 4]))
    out, lse = B.sparse_prefill_paged(cuda(q, True), cuda(k, True), cuda(v, True), cuda(logical), None,
                                      cuda(cu), cuda(kv_lens.astype(np.int32)), cuda(table), ps,
                                      1.0 / 16.0, n_pages=n_pages, union_g=G)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    O, L = oracle.sparse_prefill_paged(q, k, v, logical, None, cu, kv_lens, table, ps, 1.0 / 16.0,
                                       n_pages)
    assert_parity(out, lse, O, L, what=f"paged case {case}: reqs={n_req} ps={ps} G={G}")


@pytest.mark.parametrize("case", range(10))
def test_fuzz_mla(B, case):
    import torch
    rng = np.random.default_rng(4000 + case)
    H = int(rng.integers(1, 41))
    R, S, K = int(rng.integers(1, 120)), int(rng.integers(16, 900)), int(rng.integers(1, 400))
    G = int(rng.choice([0, 0, 2, 4]))
    q = W.randn_bf16(rng, (R, H, 576))
    kv = W.randn_bf16(rng, (S, 576))
    idx, tl = random_indices(rng, R, K, S, dup=(G == 0), junk=True)
    out, lse = B.sparse_mla_prefill(cuda(q, True), cuda(kv, True), cuda(idx),
                                    None if tl is None else cuda(tl), 1.0 / 24.0, union_g=G,
                                    n_kv_slots=S)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    O, L = oracle.sparse_mla_prefill(q, kv, idx, tl, 1.0 / 24.0, n_kv_slots=S)
    assert_parity(out, lse, O, L, what=f"mla case {case}: R={R} H={H} K={K} S={S} G={G}")
