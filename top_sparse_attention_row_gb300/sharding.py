"""Row sharding of one sparse-prefill problem over several GPUs (host logic only).

Query rows are independent and ``out`` / ``lse`` are row-partitioned, so a problem splits
into contiguous row blocks with no exchange step: every GPU holds the K/V cache replica (or
the prefix its rows can see), runs qsa_sparse_prefill on its rows, and no collective touches
the data path.  Union groups (G consecutive rows) are kept whole so every shard builds
exactly the groups the unsharded call would.
"""
from __future__ import annotations


def shard_rows(n_rows: int, world: int, rank: int, union_g: int = 1) -> tuple[int, int]:
    """[start, stop) of the rows owned by `rank`; starts are multiples of the union size."""
    if world <= 0 or not (0 <= rank < world):
        raise ValueError("bad world / rank")
    G = max(1, int(union_g))
    n_groups = -(-n_rows // G)
    per = -(-n_groups // world)
    g0 = min(rank * per, n_groups)
    g1 = min(g0 + per, n_groups)
    return min(g0 * G, n_rows), min(g1 * G, n_rows)


def sharded_prefill(q, k_cache, v_cache, indices, topk_len, scale, world, rank, union_g=0,
                    out=None, lse=None, stream=None):
    """Run this rank's row block through the C ABI; returns (start, stop, out_block, lse_block)."""
    from . import binding
    start, stop = shard_rows(q.shape[0], world, rank, max(1, union_g))
    if start == stop:
        return start, stop, None, None
    o, l = binding.sparse_prefill(
        q[start:stop], k_cache, v_cache, indices[start:stop],
        None if topk_len is None else topk_len[start:stop], scale, union_g=union_g,
        out=None if out is None else out[start:stop],
        lse=None if lse is None else lse[start:stop], stream=stream)
    return start, stop, o, l
