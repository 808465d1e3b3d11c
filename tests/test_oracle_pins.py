"""The CPU oracle against facts that do not come from the oracle (CPU only)."""
import numpy as np
import pytest

import oracle
import pins


@pytest.mark.parametrize("check", pins.ATTENTION_CHECKS, ids=lambda c: c.__name__)
def test_attention_pin(check):
    assert check(oracle.sparse_prefill) == []


def test_rows_subset_matches_full():
    q, k, v, idx, pos, scale = pins.dense_case(seed=5)
    O, L = oracle.sparse_prefill(q, k, v, idx, None, scale)
    rows = [0, 7, 19]
    Os, Ls = oracle.sparse_prefill_rows(q, k, v, idx, None, scale, rows)
    assert np.array_equal(Os, O[rows]) and np.array_equal(Ls, L[rows])


def test_bf16_bits_are_decoded_exactly():
    # 0x3F80 = 1.0, 0xC000 = -2.0, 0x3EAB ~ 0.333984375 (bf16), 0x0000 = 0
    bits = np.array([[[0x3F80, 0xC000, 0x3EAB, 0x0000]]], dtype=np.uint16)
    q = bits.copy()
    k = np.array([[[0x3F80, 0x3F80, 0x3F80, 0x3F80]]], dtype=np.uint16)
    v = bits.copy()
    O, L = oracle.sparse_prefill(q, k, v, np.array([[0]], dtype=np.int32), None, 1.0)
    assert np.array_equal(O[0, 0], [1.0, -2.0, 0.333984375, 0.0])
    assert L[0, 0] == 1.0 - 2.0 + 0.333984375


def test_union_matches_bruteforce_sets():
    assert pins.check_union_bruteforce(oracle.union_build) == []


def test_union_attention_equals_per_token():
    assert pins.check_union_attention(oracle.union_build, oracle.union_attention,
                                      oracle.sparse_prefill) == []


def test_union_contract_properties():
    idx, tl = pins.union_case(300, R=40, K=24, S=60, G=4)
    uidx, ubits, ulen = oracle.union_build(idx, tl, 4)
    for gi in range(len(ulen)):
        n = ulen[gi]
        lst = uidx[gi, :n]
        assert len(set(lst.tolist())) == n and np.all(lst >= 0)       # each slot once, no -1
        rows = range(4 * gi, min(4 * gi + 4, idx.shape[0]))
        for x, b in zip(lst, ubits[gi, :n]):
            owners = 0
            for u, r in enumerate(rows):
                L = min(max(int(tl[r]), 0), idx.shape[1])
                owners |= int(x in idx[r, :L]) << u
            assert owners == b                                         # bits = OR of owners


def test_sorted_rows_vs_python_sorted():
    idx, tl = pins.union_case(301, R=12, K=20, S=50, G=2)
    srt = oracle.sorted_rows(idx, tl)
    for r in range(idx.shape[0]):
        L = min(max(int(tl[r]), 0), idx.shape[1])
        want = sorted(int(x) for x in idx[r, :L] if x >= 0)
        assert srt[r, :len(want)].tolist() == want
        assert np.all(srt[r, len(want):] == -1)


@pytest.mark.parametrize("check", pins.PAGED_CHECKS, ids=lambda c: c.__name__)
def test_paged_pin(check):
    assert check(oracle.sparse_prefill_paged) == []


@pytest.mark.parametrize("check", pins.MLA_CHECKS, ids=lambda c: c.__name__)
def test_mla_pin(check):
    fn = lambda q, kv, idx, tl, scale, d_v: oracle.sparse_mla_prefill(q, kv, idx, tl, scale, d_v)
    assert check(fn) == []


def test_page_split_pin():
    fn = lambda src, dst, n, sps, dps, secs, mark: oracle.page_split(src, dst, n, sps, dps, secs, mark)
    assert pins.check_page_split(fn) == []


def test_page_mark_pin():
    assert pins.check_page_mark(oracle.page_mark) == []


def test_e4m3_decode_pin():
    assert pins.check_e4m3_decode(oracle.e4m3_decode) == []


def test_fp8_attention_pin():
    assert pins.check_fp8_attention(oracle.sparse_prefill_fp8) == []
