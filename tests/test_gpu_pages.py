"""Touched-page mark and masked page split (qsa_page_mark / qsa_page_split /
qsa_split_touched_pages) against the oracle, byte for byte (GPU only)."""
import numpy as np
import pytest

import oracle
from top_sparse_attention_row_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SECS = [512, 16, 128]


@pytest.fixture(scope="module")
def B():
    from top_sparse_attention_row_gb300 import build, binding
    build.build()
    binding.load_library()
    return binding


def cuda(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def small_case(seed=1, n_pages=12, src_ps=256, n_idx=(3, 40)):
    rng = np.random.default_rng(seed)
    tb = sum(SECS)
    src = rng.integers(0, 256, size=n_pages * src_ps * tb, dtype=np.uint8)
    stale = rng.integers(0, 256, size=src.size, dtype=np.uint8)
    idx = rng.integers(-2, n_pages * src_ps + 300, size=n_idx).astype(np.int32)
    idx[0, :] = -1
    return src, stale, idx


def test_page_mark_matches_oracle(B):
    import torch
    _, _, idx = small_case()
    got = B.page_mark(cuda(idx), 256, 12).cpu().numpy()
    torch.cuda.synchronize()
    assert np.array_equal(got, oracle.page_mark(idx, 256, 12))


@pytest.mark.parametrize("dst_ps", [256, 128, 64, 16])
def test_full_split_matches_oracle(B, dst_ps):
    src, stale, _ = small_case(seed=dst_ps)
    d = cuda(stale)
    B.page_split(cuda(src), d, 12, 256, dst_ps, SECS)
    got = d.cpu().numpy()
    assert np.array_equal(got, oracle.page_split(src, stale, 12, 256, dst_ps, SECS))


def test_masked_split_touches_only_marked_pages(B):
    src, stale, idx = small_case(seed=3, n_idx=(2, 6))
    mark = cuda(np.zeros(12, dtype=np.uint8))
    d = cuda(stale)
    B.split_touched_pages(cuda(idx), cuda(src), d, mark, 12, 256, 64, SECS)
    want_mark = oracle.page_mark(idx, 256, 12)
    assert np.array_equal(mark.cpu().numpy(), want_mark)
    assert 0 < want_mark.sum() < 12
    assert np.array_equal(d.cpu().numpy(), oracle.page_split(src, stale, 12, 256, 64, SECS, want_mark))


def test_split_replays_in_a_cuda_graph(B):
    """The mark + masked split captured once and replayed for new indices written in place:
    fixed grid, no host read."""
    import torch
    src, stale, idx = small_case(seed=4, n_idx=(2, 5))
    d_src, d_dst, d_idx = cuda(src), cuda(stale), cuda(idx)
    mark = cuda(np.zeros(12, dtype=np.uint8))
    B.split_touched_pages(d_idx, d_src, d_dst, mark, 12, 256, 64, SECS)     # warm-up
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        B.split_touched_pages(d_idx, d_src, d_dst, mark, 12, 256, 64, SECS, stream=s)
    idx2 = np.random.default_rng(5).integers(0, 12 * 256, size=idx.shape).astype(np.int32)
    d_dst.copy_(cuda(stale))
    d_idx.copy_(cuda(idx2))
    g.replay()
    torch.cuda.synchronize()
    want = oracle.page_split(src, stale, 12, 256, 64, SECS, oracle.page_mark(idx2, 256, 12))
    assert np.array_equal(d_dst.cpu().numpy(), want)


def test_decode_step_workload(B):
    """The benchmark's pool (4096 pages of 256 x 656 bytes, 8 requests x 512-token windows):
    touched pages against the oracle, every other page unchanged."""
    import torch
    w = W.make_page_split()
    n, sps, dps = w["n_src_pages"], w["src_page_size"], w["dst_page_size"]
    src = cuda(w["pool"])
    stale = torch.zeros_like(src)
    mark = torch.empty(n, dtype=torch.uint8, device="cuda")
    B.split_touched_pages(cuda(w["indices"]), src, stale, mark, n, sps, dps, w["section_bytes"])
    torch.cuda.synchronize()
    want_mark = oracle.page_mark(w["indices"], sps, n)
    got_mark = mark.cpu().numpy()
    assert np.array_equal(got_mark, want_mark)
    assert 8 <= want_mark.sum() <= 24
    got = stale.cpu().numpy()
    pb = sps * sum(w["section_bytes"])
    touched = np.flatnonzero(want_mark)
    # expected bytes of the touched pages only: the oracle over a pool of just those pages
    sub_src = np.concatenate([w["pool"][p * pb:(p + 1) * pb] for p in touched])
    sub_want = oracle.page_split(sub_src, np.zeros_like(sub_src), len(touched), sps, dps,
                                 w["section_bytes"])
    for k, p in enumerate(touched):
        assert np.array_equal(got[p * pb:(p + 1) * pb], sub_want[k * pb:(k + 1) * pb])
    untouched = np.ones(n, dtype=bool)
    untouched[touched] = False
    assert not got.reshape(n, pb)[untouched].any()
