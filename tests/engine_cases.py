"""Small seeded workloads shared by the gather-engine comparison (parent and child process)."""
from top_sparse_attention_row_gb300 import workloads as W


def cases():
    """(name, workload, union_g): several tiles with a ragged tail, two KV heads, a paged batch
    with per-row topk_len, and a union group of 2 over a random walk."""
    return [
        ("chunk6", W.make_chunk(n_rows=96, context=2200, n_qheads=6, n_kvheads=1, topk=2051,
                                seed=11, name="chunk6"), 0),
        ("chunk24", W.make_chunk(n_rows=40, context=1800, n_qheads=24, n_kvheads=2, topk=1000,
                                 seed=12, name="chunk24"), 0),
        ("mixed", W.make_mixed(new_tokens=(64, 130), prefixes=(0, 2000), page_size=64), 0),
        ("union2", W.make_union(n_rows=300, topk=256), 2),
    ]
