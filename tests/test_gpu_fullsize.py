"""Full-size workloads in the benchmark's launch configuration, checked on sampled rows
against the oracle (GPU only)."""
import numpy as np
import pytest

import oracle
from helpers import to_device, assert_parity
from top_sparse_attention_row_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from top_sparse_attention_row_gb300 import build, binding
    build.build()
    binding.load_library()
    return binding


def sample_rows(n, k=40, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(n, size=min(k, n), replace=False).tolist()) | {0, 1, n - 2, n - 1}
    return np.array(sorted(rows))


@pytest.mark.parametrize("name,union_g", [
    ("group6_32k", 0),
    ("group12_128k", 0),
    ("group12_128k_12q1kv", 0),
    ("union_8k", 0), ("union_8k", 2), ("union_8k", 4),
    ("mixed_paged", 0),
])
def test_full_size_sampled(B, name, union_g):
    import torch
    w = W.make(name)
    q, k, v, idx, tl = to_device(w)
    out, lse = B.sparse_prefill(q, k, v, idx, tl, w.scale, union_g=union_g)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    rows = sample_rows(w.n_rows, seed=union_g)
    if name == "union_8k":       # include the walk's start and group boundaries
        rows = np.unique(np.concatenate([rows, [2046, 2047, 2048, 2049, 4095, 4096]]))
    O, L = oracle.sparse_prefill_rows(w.q, w.k, w.v, w.indices, w.topk_len, w.scale, rows)
    assert_parity(out, lse, O, L, rows=rows, what=f"{name} G={union_g}")
    # properties that hold at any size: finite output, LSE finite for rows with a slot
    o = out.float()
    assert torch.isfinite(o).all()
    assert torch.isfinite(lse[torch.from_numpy(w.valid_counts() > 0).cuda()]).all()
