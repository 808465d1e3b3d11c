"""The product's row-sharding path on one GPU: sharding.sharded_prefill runs every rank's row block
through the C ABI, one shard after another, into slices of one output; the assembled result is
bit-identical to the unsharded call where a shard runs the same geometry (rows are independent
and union groups stay whole; a small shard may split its rows over clusters, which sums in another
order) and matches the oracle row by row (GPU only)."""
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


@pytest.mark.parametrize("world", [2, 3, 8])
@pytest.mark.parametrize("G", [0, 4])
def test_sharded_prefill_assembles_the_unsharded_result(B, world, G):
    import torch
    from top_sparse_attention_row_gb300.sharding import sharded_prefill, shard_rows
    w = W.make_union(n_rows=613, topk=300)               # ragged last group at G = 4
    q, k, v, idx, tl = to_device(w)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.n_rows, w.n_qheads), float("nan"), dtype=torch.float32, device="cuda")
    covered = 0
    for rank in range(world):
        a, b, o, l = sharded_prefill(q, k, v, idx, tl, w.scale, world, rank, union_g=G, out=out, lse=lse)
        assert (a, b) == shard_rows(w.n_rows, world, rank, max(1, G))
        covered += b - a
    torch.cuda.synchronize()
    assert covered == w.n_rows and B.device_status() == 0
    ref_out, ref_lse = B.sparse_prefill(q, k, v, idx, tl, w.scale, union_g=G)
    torch.cuda.synchronize()
    # A shard whose rows are few enough for split items (a cluster per row, merged partials)
    # sums each row in another order than the unsharded call: bit-identical rows are expected
    # only from shards that run the unsharded call's geometry.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    full_split = B.select_geometry(w.n_qheads, w.n_kvheads, G, w.topk, 256, w.n_rows, sms)["split"]
    for rank in range(world):
        a, b = shard_rows(w.n_rows, world, rank, max(1, G))
        if a == b:
            continue
        split = B.select_geometry(w.n_qheads, w.n_kvheads, G, w.topk, 256, b - a, sms)["split"]
        if split == full_split:
            assert torch.equal(out[a:b].view(torch.int16), ref_out[a:b].view(torch.int16))
            assert torch.equal(lse[a:b], ref_lse[a:b])
        else:
            assert float((out[a:b].float() - ref_out[a:b].float()).abs().max()) <= 2e-2
    O, L = oracle.sparse_prefill(w.q, w.k, w.v, w.indices, w.topk_len, w.scale)
    assert_parity(out, lse, O, L, what=f"sharded world={world} G={G}")
