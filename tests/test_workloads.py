"""Seeded synthetic workloads: shapes, determinism and the structure the pages describe."""
import numpy as np
import pytest

from top_sparse_attention_row_gb300 import workloads as W


def test_bf16_round_trip_and_rounding():
    x = np.array([1.0, -2.5, 3.0e-3, 1.00390625, 1.005859375], dtype=np.float32)
    b = W.f32_to_bf16_bits(x)
    y = W.bf16_to_f32(b)
    assert y[0] == 1.0 and y[1] == -2.5
    assert y[3] == 1.0                   # 1 + 2^-8 is a tie -> even (1.0)
    assert y[4] == 1.0078125             # 1 + 3*2^-9 rounds up to 1 + 2^-7
    assert np.all(np.abs(y - x) <= np.abs(x) * 2.0 ** -8)


def test_tiny_config_shape_and_causality():
    w = W.make_tiny()
    assert w.q.shape == (256, 6, 256) and w.k.shape == (512, 1, 256) and w.indices.shape == (256, 128)
    assert w.topk_len is None and w.scale == 1.0 / 16.0
    for r in range(w.n_rows):
        p = w.positions[r]
        row = w.indices[r]
        assert np.all(row >= 0) and np.all(row <= p) and len(set(row.tolist())) == 128
    w2 = W.make_tiny()
    assert np.array_equal(w.q, w2.q) and np.array_equal(w.indices, w2.indices)


def test_causal_uniform_short_prefix_pads():
    rng = np.random.default_rng(0)
    idx = W.causal_uniform_indices(rng, np.array([0, 3, 10]), 6)
    assert sorted(idx[0][idx[0] >= 0].tolist()) == [0] and np.sum(idx[0] < 0) == 5
    assert sorted(idx[1][idx[1] >= 0].tolist()) == [0, 1, 2, 3]
    assert len(set(idx[2].tolist())) == 6 and idx[2].max() <= 10


def test_random_walk_structure():
    K, R = 64, 400
    idx = W.random_walk_indices(np.random.default_rng(3), R, K)
    for t in range(K):
        assert sorted(idx[t][idx[t] >= 0].tolist()) == list(range(t + 1))
    n_swap = max(1, round(0.02 * K))
    for t in range(K, R):
        row, prev = idx[t], idx[t - 1]
        assert len(set(row.tolist())) == K and row.max() <= t and row.min() >= 0
        changed = int(np.sum(row != prev))
        assert changed == min(n_swap, t + 1 - K)


def test_union_calibration_band():
    """The walk's union sizes sit inside the band the pages measured on captures
    (G=2: 1.00-1.12x, G=4: 1.01-1.23x)."""
    idx = W.random_walk_indices(np.random.default_rng(3), 2048 + 512, 2048)
    r2 = W.union_size_ratio(idx, 2, start_row=2048)
    r4 = W.union_size_ratio(idx, 4, start_row=2048)
    assert 1.0 <= r2 <= 1.12 and 1.01 <= r4 <= 1.23, (r2, r4)


def test_mixed_paged_translation():
    w = W.make_mixed(new_tokens=(8, 40, 16), prefixes=(0, 100, 64), page_size=16, topk=32)
    m = w.meta
    assert w.n_rows == 64 and w.n_slots == sum(-(-L // 16) for L in m["kv_lens"]) * 16
    # every physical page belongs to exactly one request
    allp = np.concatenate(m["page_tables"])
    assert sorted(allp.tolist()) == list(range(len(allp)))
    for r in range(w.n_rows):
        i = m["req_of_row"][r]
        p = w.positions[r]
        n = w.topk_len[r]
        assert n == min(p + 1, 32) and np.all(w.indices[r, n:] == -1)
        phys = w.indices[r, :n]
        page, off = phys // 16, phys % 16
        inv = {int(pg): j for j, pg in enumerate(m["page_tables"][i])}
        logical = np.array([inv[int(pg)] * 16 + o for pg, o in zip(page, off)])
        assert np.all(logical <= p) and len(set(logical.tolist())) == n


@pytest.mark.slow
def test_full_size_configs_shapes():
    w = W.make_group6()
    assert w.indices.shape == (8192, 2051) and np.all(w.indices >= 0)
    assert w.k.shape == (32768, 1, 256) and w.positions[0] == 24576
