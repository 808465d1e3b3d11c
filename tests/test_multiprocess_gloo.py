"""The N > 1 path on CPU: world_size-2 gloo ranks shard rows (union groups whole), each computes
its block, and the gathered result equals the single-process result; the benchmark's
max-over-ranks reduction works over gloo."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as tmp

from top_sparse_attention_row_gb300.sharding import shard_rows


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_shard_rows_cover_and_keep_groups():
    for n in (1, 7, 256, 613, 8192):
        for world in (1, 2, 3, 8):
            for G in (1, 2, 4, 8):
                spans = [shard_rows(n, world, r, G) for r in range(world)]
                assert spans[0][0] == 0 and spans[-1][1] == n
                for (a, b), (c, d) in zip(spans, spans[1:]):
                    assert b == c
                for a, b in spans:
                    assert (a % G == 0 or a == b == n) and a <= b


def _worker(rank, world, port, G, result_path):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    sys.path.insert(0, os.path.join(root, "tests"))
    import oracle
    import bench
    from top_sparse_attention_row_gb300 import workloads as W
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        w = W.make_chunk(n_rows=61, context=400, n_qheads=6, n_kvheads=1, topk=64, seed=3, name="shard")
        a, b = shard_rows(w.n_rows, world, rank, G)
        rows = np.arange(a, b)
        if G > 1:
            uidx, ubits, ulen = oracle.union_build(w.indices[a:b], None, G)
            O, L = oracle.union_attention(w.q[a:b], w.k, w.v, uidx, ubits, ulen, G, w.scale)
        else:
            O, L = oracle.sparse_prefill_rows(w.q, w.k, w.v, w.indices, None, w.scale, rows)
        pad = w.n_rows
        buf = torch.zeros((pad, 6, 256), dtype=torch.float64)
        lbuf = torch.full((pad, 6), float("nan"), dtype=torch.float64)
        buf[: b - a] = torch.from_numpy(O)
        lbuf[: b - a] = torch.from_numpy(L)
        outs = [torch.zeros_like(buf) for _ in range(world)]
        lses = [torch.zeros_like(lbuf) for _ in range(world)]
        dist.all_gather(outs, buf)
        dist.all_gather(lses, lbuf)
        t = bench.max_over_ranks([float(rank + 1), 10.0 * (world - rank)], torch.device("cpu"))
        if rank == 0:
            full_O, full_L = oracle.sparse_prefill(w.q, w.k, w.v, w.indices, None, w.scale)
            got_O = np.concatenate([outs[r][: shard_rows(w.n_rows, world, r, G)[1] - shard_rows(w.n_rows, world, r, G)[0]].numpy() for r in range(world)])
            got_L = np.concatenate([lses[r][: shard_rows(w.n_rows, world, r, G)[1] - shard_rows(w.n_rows, world, r, G)[0]].numpy() for r in range(world)])
            ok = (np.max(np.abs(got_O - full_O)) < 1e-12 and np.max(np.abs(got_L - full_L)) < 1e-12
                  and t == [float(world), 10.0 * world])
            with open(result_path, "w") as f:
                f.write("ok" if ok else f"mismatch {t}")
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("G", [1, 4])
def test_two_rank_gloo_sharding(tmp_path, G):
    path = str(tmp_path / "result.txt")
    tmp.spawn(_worker, args=(2, _free_port(), G, path), nprocs=2, join=True)
    assert open(path).read() == "ok"
