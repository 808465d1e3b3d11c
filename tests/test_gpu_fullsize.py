"""Full-size workloads in the benchmark's launch configuration, every row checked against the
oracle (GPU only).  The oracle runs in spawned worker processes over the host cores; a failure
names the worst row.  The union lists and bits of the full-size union workload are compared
bit for bit as well."""
import numpy as np
import pytest

from helpers import to_device
from top_sparse_attention_row_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from top_sparse_attention_row_gb300 import build, binding
    build.build()
    binding.load_library()
    return binding


@pytest.mark.parametrize("name,union_g", [
    ("tiny", 0),
    ("group6_32k", 0),
    ("group12_128k", 0),
    ("group12_128k_12q1kv", 0),
    ("union_8k", 0), ("union_8k", 2), ("union_8k", 4),
    ("mixed_paged", 0), ("mixed_paged", 4),
])
def test_full_size_every_row(B, oracle_pool, name, union_g):
    import torch
    w = W.make(name)
    q, k, v, idx, tl = to_device(w)
    out, lse = B.sparse_prefill(q, k, v, idx, tl, w.scale, union_g=union_g)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    assert torch.isfinite(out.float()).all()
    oracle_pool.check_all_rows((name, ""), "plain", out, lse, f"{name} G={union_g}")


@pytest.mark.parametrize("G", [2, 4])
def test_union_build_full_size_bit_exact(B, oracle_pool, G):
    """The union lists, ownership bits and lengths of the 8192-row, topk-2048 random walk, as the
    benchmark's union calls build them, against the oracle for every group."""
    import torch
    w = W.make("union_8k")
    _, _, _, idx, tl = to_device(w)
    _, uidx, ubits, ulen = B.union_build(idx, tl, G, want_sorted=False)
    torch.cuda.synchronize()
    oracle_pool.check_union_build(("union_8k", ""), G, uidx.cpu().numpy(), ubits.cpu().numpy(),
                                  ulen.cpu().numpy(), f"union_8k G={G}")
