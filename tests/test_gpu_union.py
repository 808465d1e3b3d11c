"""Union mode on the GPU: union lists / bits / sorted rows bit-exact against the oracle, and
union attention (G = 2, 4, 8 and odd G, with a partial last group) against per-token oracle
output (GPU only)."""
import numpy as np
import pytest

import oracle
import pins
from helpers import to_device, assert_parity
from top_sparse_attention_row_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from top_sparse_attention_row_gb300 import build, binding
    build.build()
    binding.load_library()
    return binding


def _dev(a):
    import torch
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


@pytest.mark.parametrize("G", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("with_len", [False, True])
@pytest.mark.parametrize("want_sorted", [True, False])     # bitonic kernel / bitmap kernel
def test_union_build_bit_exact(B, G, with_len, want_sorted):
    import torch
    idx, tl = pins.union_case(400 + G, R=37, K=40, S=90, G=G, with_len=with_len)
    srt, uidx, ubits, ulen = B.union_build(_dev(idx), _dev(tl), G, want_sorted=want_sorted)
    torch.cuda.synchronize()
    e_idx, e_bits, e_len = oracle.union_build(idx, tl, G)
    if want_sorted:
        assert np.array_equal(srt.cpu().numpy(), oracle.sorted_rows(idx, tl))
    assert np.array_equal(ulen.cpu().numpy(), e_len)
    assert np.array_equal(uidx.cpu().numpy(), e_idx)
    assert np.array_equal(ubits.cpu().numpy(), e_bits)


@pytest.mark.parametrize("S", [1 << 17, 600_000, 5_000_000])
def test_union_build_wide_slot_ranges(B, S):
    """Slot numbers beyond one bitmap window (131072 slots) take several windows; a slot
    count filter also applies."""
    import torch
    rng = np.random.default_rng(S)
    R, K, G = 45, 300, 4
    base = rng.choice(S, size=K, replace=False)
    idx = np.stack([np.where(rng.random(K) < 0.3, rng.integers(0, S, size=K), base) for _ in range(R)]).astype(np.int32)
    idx[rng.random(idx.shape) < 0.05] = -1
    for n_slots in (0, S // 2):
        _, uidx, ubits, ulen = B.union_build(_dev(idx), None, G, n_kv_slots=n_slots, want_sorted=False)
        torch.cuda.synchronize()
        e_idx, e_bits, e_len = oracle.union_build(idx, None, G, n_kv_slots=n_slots)
        assert np.array_equal(ulen.cpu().numpy(), e_len)
        assert np.array_equal(uidx.cpu().numpy(), e_idx)
        assert np.array_equal(ubits.cpu().numpy(), e_bits)


def test_union_build_walk_bit_exact(B):
    import torch
    idx = W.random_walk_indices(np.random.default_rng(5), 700, 512)
    for G in (2, 4):
        srt, uidx, ubits, ulen = B.union_build(_dev(idx), None, G, want_sorted=False)
        torch.cuda.synchronize()
        e_idx, e_bits, e_len = oracle.union_build(idx, None, G)
        assert np.array_equal(ulen.cpu().numpy(), e_len)
        assert np.array_equal(uidx.cpu().numpy(), e_idx)
        assert np.array_equal(ubits.cpu().numpy(), e_bits)


def _walk_workload(n_rows, topk, hq=8, hkv=1, seed=21):
    rng = np.random.default_rng(seed)
    q = W.randn_bf16(rng, (n_rows, hq, 256))
    k = W.randn_bf16(rng, (n_rows, hkv, 256))
    v = W.randn_bf16(rng, (n_rows, hkv, 256))
    idx = W.random_walk_indices(rng, n_rows, topk)
    return W.Workload("walk", q, k, v, idx, None, 1.0 / 16.0, np.arange(n_rows))


@pytest.mark.parametrize("G", [1, 2, 4, 8, 3])
def test_union_attention_matches_per_token_oracle(B, G):
    import torch
    w = _walk_workload(n_rows=613, topk=384)          # 613 % G != 0 for G = 2, 4, 8, 3
    q, k, v, idx, tl = to_device(w)
    B.reset_counters()
    out, lse = B.sparse_prefill(q, k, v, idx, tl, w.scale, union_g=G)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    c = B.counters()
    # the selector decides whether the G x 8-head union tile fits; a misfit is a counted fallback
    legal = B.select_geometry(8, 1, G, 384, 256, 613)["union_g"] > 1
    assert c["calls_union"] == (1 if (G > 1 and legal) else 0)
    assert c["union_fallbacks"] == (1 if (G > 1 and not legal) else 0)
    O, L = oracle.sparse_prefill(w.q, w.k, w.v, w.indices, None, w.scale)
    assert_parity(out, lse, O, L, what=f"union G={G}")


def test_union_with_two_kv_heads_and_topk_len(B):
    import torch
    rng = np.random.default_rng(8)
    R, K, S = 203, 200, 500
    idx, tl = pins.union_case(9, R=R, K=K, S=S, G=4, dup=False)
    w = W.Workload("u2", W.randn_bf16(rng, (R, 8, 256)), W.randn_bf16(rng, (S, 2, 256)),
                   W.randn_bf16(rng, (S, 2, 256)), idx, tl, 0.0625, np.arange(R))
    q, k, v, idx_d, tl_d = to_device(w)
    for G in (2, 4):
        out, lse = B.sparse_prefill(q, k, v, idx_d, tl_d, w.scale, union_g=G)
        torch.cuda.synchronize()
        O, L = oracle.sparse_prefill(w.q, w.k, w.v, idx, tl, w.scale)
        assert_parity(out, lse, O, L, what=f"union 2 kv heads G={G}")


def test_union_fallback_is_counted_and_exact(B):
    import torch
    rng = np.random.default_rng(10)
    R, K, S = 64, 128, 300
    idx, _ = pins.union_case(11, R=R, K=K, S=S, G=4, dup=False, with_len=False)
    w = W.Workload("fb", W.randn_bf16(rng, (R, 32, 256)), W.randn_bf16(rng, (S, 1, 256)),
                   W.randn_bf16(rng, (S, 1, 256)), idx, None, 0.0625, np.arange(R))
    q, k, v, idx_d, tl_d = to_device(w)
    B.reset_counters()
    out, lse = B.sparse_prefill(q, k, v, idx_d, None, w.scale, union_g=4)   # 4 x 32 > 64 columns
    torch.cuda.synchronize()
    c = B.counters()
    assert c["union_fallbacks"] == 1 and c["calls_per_token"] == 1
    O, L = oracle.sparse_prefill(w.q, w.k, w.v, idx, None, w.scale)
    assert_parity(out, lse, O, L, what="union fallback")


def test_union_caller_workspace(B):
    import torch
    w = _walk_workload(n_rows=300, topk=256, seed=31)
    q, k, v, idx, tl = to_device(w)
    nbytes = B.workspace_bytes(w.n_rows, w.topk, 4)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out, lse = B.sparse_prefill(q, k, v, idx, None, w.scale, union_g=4, workspace=ws)
    torch.cuda.synchronize()
    O, L = oracle.sparse_prefill(w.q, w.k, w.v, w.indices, None, w.scale)
    assert_parity(out, lse, O, L, what="caller workspace")
    with pytest.raises(RuntimeError, match="WORKSPACE"):
        B.sparse_prefill(q, k, v, idx, None, w.scale, union_g=4, workspace=ws[: nbytes // 2])
