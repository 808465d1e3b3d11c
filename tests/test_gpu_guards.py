"""Memory-safety checks that stand in for compute-sanitizer (GPU only):
  * guard bands -- every output (O, LSE, union workspace, split pool) sits between 64 KiB of
    canary bytes inside a larger allocation, and each entry point must leave the canaries intact
    while its payload still matches the oracle;
  * 64-bit addressing -- a batch whose O offsets pass 2^31 elements ("DSA prefill ...
    triton_sparse_mla", Robustness: offsets into the token rows are computed in 64 bits, so a big
    batch with 64 or 128 heads never aliases a neighbouring token's output);
  * the union tail the pages single out: T = 1023 rows at G = 4."""
import numpy as np
import pytest

import oracle
from helpers import to_device, assert_parity
from top_sparse_attention_row_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GUARD = 64 * 1024          # bytes of canary on each side
CANARY = 0xA5


@pytest.fixture(scope="module")
def B():
    from top_sparse_attention_row_gb300 import build, binding
    build.build()
    binding.load_library()
    return binding


class Guarded:
    """A tensor of `shape`/`dtype` carved out of a byte buffer with canary bands around it."""

    def __init__(self, shape, dtype):
        import torch
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.n = n
        self.raw = torch.full((GUARD + n + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(*shape)

    def intact(self):
        import torch
        torch.cuda.synchronize()
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.n:]
        return bool((head == CANARY).all()) and bool((tail == CANARY).all())


def test_guards_per_token_union_and_workspace(B):
    import torch
    w = W.make_union(n_rows=301, topk=256)
    q, k, v, idx, tl = to_device(w)
    O, L = oracle.sparse_prefill(w.q, w.k, w.v, w.indices, w.topk_len, w.scale)
    for G in (0, 4):
        out = Guarded(tuple(q.shape), torch.bfloat16)
        lse = Guarded((w.n_rows, w.n_qheads), torch.float32)
        ws = Guarded((max(B.workspace_bytes(w.n_rows, w.topk, G), 256),), torch.uint8) if G else None
        B.sparse_prefill(q, k, v, idx, tl, w.scale, out=out.t, lse=lse.t, union_g=G,
                         workspace=None if ws is None else ws.t)
        torch.cuda.synchronize()
        assert B.device_status() == 0
        assert out.intact() and lse.intact() and (ws is None or ws.intact()), f"G={G}"
        assert_parity(out.t, lse.t, O, L, what=f"guarded G={G}")


def test_guards_paged_fp8_and_mla(B):
    import torch
    # paged
    w = W.make_mixed(new_tokens=(40, 70), prefixes=(0, 900), page_size=64)
    m = w.meta
    q, k, v, _, tl = to_device(w)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    out = Guarded(tuple(q.shape), torch.bfloat16)
    lse = Guarded((w.n_rows, w.n_qheads), torch.float32)
    B.sparse_prefill_paged(q, k, v, i32(m["logical_indices"]), tl, i32(m["cu_seqlens_q"]),
                           i32(m["kv_lens_array"]), i32(m["page_table"]), m["page_size"], w.scale,
                           n_pages=m["n_pages"], out=out.t, lse=lse.t)
    assert out.intact() and lse.intact()
    O, L = oracle.sparse_prefill(w.q, w.k, w.v, w.indices, w.topk_len, w.scale)
    assert_parity(out.t, lse.t, O, L, what="guarded paged")
    # FP8
    wf = W.with_fp8_cache(w, 64)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = Guarded(tuple(q.shape), torch.bfloat16)
    lse = Guarded((w.n_rows, w.n_qheads), torch.float32)
    idx = i32(w.indices)
    B.sparse_prefill_fp8(q, t(wf.meta["k8"]), t(wf.meta["v8"]), t(wf.meta["k_scale"]),
                         t(wf.meta["v_scale"]), 64, idx, tl, w.scale, out=out.t, lse=lse.t)
    assert out.intact() and lse.intact()
    # MLA, per-token and union
    wm = W.make_mla(seed=81, n_rows=200, topk=256, n_heads=8, name="mla_guard")
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    qm, kvm, im = bf(wm.q), bf(wm.k.reshape(wm.k.shape[0], -1)), i32(wm.indices)
    Om, Lm = oracle.sparse_mla_prefill(wm.q, wm.k.reshape(wm.k.shape[0], -1), wm.indices, None, wm.scale)
    for G in (0, 4):
        out = Guarded((wm.n_rows, 8, 512), torch.bfloat16)
        lse = Guarded((wm.n_rows, 8), torch.float32)
        B.sparse_mla_prefill(qm, kvm, im, None, wm.scale, out=out.t, lse=lse.t, union_g=G)
        assert out.intact() and lse.intact(), f"MLA G={G}"
        assert_parity(out.t, lse.t, Om, Lm, what=f"guarded MLA G={G}")
    assert B.device_status() == 0


def test_guards_page_split(B):
    import torch
    rng = np.random.default_rng(83)
    secs, n_pages, sps = [512, 16, 128], 10, 256
    src = rng.integers(0, 256, size=n_pages * sps * sum(secs), dtype=np.uint8)
    dst = Guarded((src.size,), torch.uint8)
    dst.t.zero_()
    mark = Guarded((n_pages,), torch.uint8)
    idx = rng.integers(-1, n_pages * sps, size=(2, 7)).astype(np.int32)
    B.split_touched_pages(torch.from_numpy(idx).cuda(), torch.from_numpy(src).cuda(), dst.t, mark.t,
                          n_pages, sps, 64, secs)
    assert dst.intact() and mark.intact()
    want = oracle.page_split(src, np.zeros_like(src), n_pages, sps, 64, secs,
                             oracle.page_mark(idx, sps, n_pages))
    assert np.array_equal(dst.t.cpu().numpy(), want)


def test_offsets_past_two_to_the_31_elements(B):
    """33000 rows x 256 query heads x 256 dims: O and q offsets of the last rows exceed 2^31
    elements (4.3 GB each); sampled rows at both ends against the oracle."""
    import torch
    rng = np.random.default_rng(84)
    R, Hq, Hkv, S, K = 33000, 256, 2, 4096, 64
    assert (R - 1) * Hq * 256 > 2 ** 31
    kv_shape = (S, Hkv, 256)
    k = W.randn_bf16(rng, kv_shape)
    v = W.randn_bf16(rng, kv_shape)
    idx = rng.integers(-1, S, size=(R, K)).astype(np.int32)
    q = torch.randn(R, Hq, 256, device="cuda", dtype=torch.bfloat16,
                    generator=torch.Generator(device="cuda").manual_seed(85))
    dk = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).cuda()
    dv = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).cuda()
    out, lse = B.sparse_prefill(q, dk, dv, torch.from_numpy(idx).cuda(), None, 1.0 / 16.0)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    rows = np.array([0, 1, R // 2, R - 3, R - 2, R - 1])
    q_rows = q[torch.from_numpy(rows).cuda()].view(torch.int16).cpu().numpy().view(np.uint16)
    O, L = oracle.sparse_prefill_rows(q_rows, k, v, idx[rows], None, 1.0 / 16.0, np.arange(len(rows)))
    got_o = out[torch.from_numpy(rows).cuda()]
    got_l = lse[torch.from_numpy(rows).cuda()]
    assert_parity(got_o, got_l, O, L, what="64-bit offsets")


def test_union_tail_1023_rows_group_4(B):
    """The pages' tail case: 1023 rows at G = 4 leave a last group of three rows."""
    import torch
    w = W.make_union(n_rows=1023, topk=256)
    q, k, v, idx, tl = to_device(w)
    out, lse = B.sparse_prefill(q, k, v, idx, tl, w.scale, union_g=4)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    O, L = oracle.sparse_prefill(w.q, w.k, w.v, w.indices, w.topk_len, w.scale)
    assert_parity(out, lse, O, L, what="T=1023, G=4")
    tail = np.arange(1020, 1023)
    out1, lse1 = B.sparse_prefill(q, k, v, idx, tl, w.scale, union_g=0)
    torch.cuda.synchronize()
    assert_parity(out[1020:], lse[1020:], O[tail], L[tail], what="tail rows")
    assert_parity(out1[1020:], lse1[1020:], O[tail], L[tail], what="tail rows, per-token")
