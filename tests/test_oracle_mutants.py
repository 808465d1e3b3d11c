"""Each copy of the oracle below carries one planted mistake; the pins must catch every one.

The mutants are written here, on the CPU, from the oracle's definition; nothing runs on a GPU.
"""
import numpy as np
import pytest

import oracle
import pins
from oracle.attention import _as_f64, valid_slots


def _make(kv_map="div", scale_pow=1, lse_mode="full", normalize=True, honor_len=True,
          neg_is_pad=True, transpose_kv=False):
    def fn(q, k, v, indices, topk_len, scale, n_kv_slots=0):
        R, Hq, D = q.shape
        Hkv = k.shape[1]
        g = Hq // Hkv
        O = np.zeros((R, Hq, D))
        L = np.full((R, Hq), -np.inf)
        for r in range(R):
            tl = topk_len[r] if (topk_len is not None and honor_len) else None
            if neg_is_pad:
                J = valid_slots(indices[r], tl, n_kv_slots)
            else:
                row = np.asarray(indices[r][: (len(indices[r]) if tl is None else int(tl))], np.int64)
                J = row[row != -1]
            for h in range(Hq):
                kvh = h // g if kv_map == "div" else h % Hkv
                if len(J) == 0:
                    continue
                qs = _as_f64(q[r, h])
                ks = _as_f64(k[J, kvh])
                vs = _as_f64(v[J, kvh]) if not transpose_kv else _as_f64(k[J, kvh])
                s = (scale ** scale_pow) * (ks @ qs)
                m = s.max()
                p = np.exp(s - m)
                l = p.sum()
                O[r, h] = (p @ vs) / (l if normalize else 1.0)
                L[r, h] = (m + np.log(l)) if lse_mode == "full" else np.log(l)
        return O, L
    return fn


MUTANTS = {
    "kv_head_h_mod_hkv": _make(kv_map="mod"),
    "scale_applied_twice": _make(scale_pow=2),
    "lse_drops_max": _make(lse_mode="no_max"),
    "output_not_normalised": _make(normalize=False),
    "topk_len_ignored": _make(honor_len=False),
    "only_minus_one_is_padding": _make(neg_is_pad=False),
    "value_operand_swapped_for_key": _make(transpose_kv=True),
}


def test_unmutated_copy_passes():
    fn = _make()
    fails = [f for c in pins.ATTENTION_CHECKS for f in c(fn)]
    assert fails == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_attention_mutant_is_caught(name):
    fn = MUTANTS[name]
    fails = [f for c in pins.ATTENTION_CHECKS for f in c(fn)]
    assert fails, f"mutant {name} passed every pin"


def _union_mutant(kind):
    def build(indices, topk_len, G, n_kv_slots=0):
        uidx, ubits, ulen = oracle.union_build(indices, topk_len, G, n_kv_slots)
        if kind == "no_self_bit":
            # clear the emitting row's own bit where another row also owns the slot
            for gi in range(len(ulen)):
                for j in range(ulen[gi]):
                    b = int(ubits[gi, j])
                    low = b & -b
                    if b != low:
                        ubits[gi, j] = b ^ low
        elif kind == "keeps_minus_one":
            for gi in range(len(ulen)):
                if ulen[gi] < uidx.shape[1]:
                    uidx[gi, ulen[gi]] = -1
                    ubits[gi, ulen[gi]] = 1
                    ulen[gi] += 1
        elif kind == "descending_order":
            for gi in range(len(ulen)):
                n = ulen[gi]
                uidx[gi, :n] = uidx[gi, :n][::-1]
                ubits[gi, :n] = ubits[gi, :n][::-1]
        return uidx, ubits, ulen
    return build


@pytest.mark.parametrize("kind", ["no_self_bit", "keeps_minus_one", "descending_order"])
def test_union_mutant_is_caught(kind):
    assert pins.check_union_bruteforce(_union_mutant(kind))


def _paged_mutant(kind):
    """A copy of the paged oracle's translation with one planted mistake."""
    from oracle.attention import sparse_prefill_rows

    def translate(indices, cu, kv_lens, table, ps, n_pages):
        idx = np.asarray(indices, dtype=np.int64)
        table = np.asarray(table, dtype=np.int64)
        cu = np.asarray(cu, dtype=np.int64)
        out = np.full(idx.shape, -1, dtype=np.int64)
        for r in range(idx.shape[0]):
            cands = [i for i in range(len(cu) - 1) if cu[i] <= r]
            i = cands[0] if kind == "first_request_not_last" else cands[-1]
            if kind == "next_request" and i + 1 < len(cu) - 1:
                i += 1
            for j, x in enumerate(idx[r]):
                if x < 0:
                    continue
                if kv_lens is not None and kind != "kv_lens_ignored" and x >= kv_lens[i]:
                    continue
                page = x // ps
                if page >= table.shape[1]:
                    continue
                pid = table[i, page]
                if pid < 0 or (n_pages > 0 and pid >= n_pages and kind != "n_pages_ignored"):
                    continue
                off = (x // ps) % ps if kind == "offset_from_page" else x % ps
                out[r, j] = pid * ps + off
        return out

    def fn(q, kc, vc, indices, topk_len, cu, kv_lens, table, ps, scale, n_pages=0):
        phys = translate(indices, cu, kv_lens, table, ps, n_pages)
        return sparse_prefill_rows(q, kc, vc, phys, topk_len, scale, np.arange(q.shape[0]))
    return fn


def test_paged_unmutated_copy_passes():
    fn = _paged_mutant("none")
    assert [f for c in pins.PAGED_CHECKS for f in c(fn)] == []


@pytest.mark.parametrize("kind", ["first_request_not_last", "next_request", "kv_lens_ignored",
                                  "n_pages_ignored", "offset_from_page"])
def test_paged_mutant_is_caught(kind):
    fn = _paged_mutant(kind)
    assert [f for c in pins.PAGED_CHECKS for f in c(fn)], f"mutant {kind} passed every pin"


def _mla_mutant(kind):
    """A copy of the MLA oracle with one planted mistake."""
    def fn(q, kv, idx, tl, scale, d_v):
        R, H, D = q.shape
        O = np.zeros((R, H, d_v))
        L = np.full((R, H), -np.inf)
        for r in range(R):
            J = valid_slots(idx[r], None if tl is None else tl[r])
            if len(J) == 0:
                continue
            rows = np.asarray(kv, dtype=np.float64)[J]
            keys = rows[:, :d_v] if kind == "key_drops_rope" else rows
            vals = rows[:, D - d_v:] if kind == "value_from_tail" else rows[:, :d_v]
            for h in range(H):
                qh = np.asarray(q[r, 0 if kind == "head_zero_for_all" else h], dtype=np.float64)
                qk = qh[:d_v] if kind == "key_drops_rope" else qh
                s = scale * (keys @ qk)
                m = s.max()
                p = np.exp(s - m)
                O[r, h] = (p @ vals) / p.sum()
                L[r, h] = m + np.log(p.sum())
        return O, L
    return fn


def test_mla_unmutated_copy_passes():
    assert [f for c in pins.MLA_CHECKS for f in c(_mla_mutant("none"))] == []


@pytest.mark.parametrize("kind", ["key_drops_rope", "value_from_tail", "head_zero_for_all"])
def test_mla_mutant_is_caught(kind):
    assert [f for c in pins.MLA_CHECKS for f in c(_mla_mutant(kind))], f"mutant {kind} passed"


def _split_mutant(kind):
    def split(src, dst, n_pages, src_ps, dst_ps, secs, mark):
        ratio = src_ps // dst_ps
        out = np.array(dst, copy=True)
        dpb = dst_ps * sum(secs)
        for p in range(n_pages):
            if mark is not None and not mark[p]:
                continue
            for i in range(ratio):
                q = p * ratio + i
                ii = ratio - 1 - i if kind == "sub_page_reversed" else i
                order = list(range(len(secs)))
                if kind == "sections_swapped":
                    order = order[::-1]
                off = q * dpb
                for k in order:
                    sb = secs[k]
                    soff = p * src_ps * sum(secs) + src_ps * sum(secs[:k]) + ii * dst_ps * sb
                    out[off:off + dst_ps * sb] = src[soff:soff + dst_ps * sb]
                    off += dst_ps * sb
        return out
    return split


@pytest.mark.parametrize("kind", ["sub_page_reversed", "sections_swapped"])
def test_page_split_mutant_is_caught(kind):
    assert pins.check_page_split(_split_mutant(kind))


def test_page_split_unmutated_copy_passes():
    assert pins.check_page_split(_split_mutant("none")) == []


def test_page_mark_mutant_is_caught():
    def mark(idx, ps, n):                       # off by one: page (t + 1) // ps
        m = np.zeros(n, dtype=np.uint8)
        for t in np.asarray(idx).reshape(-1):
            if t >= 0 and (t + 1) // ps < n:
                m[(t + 1) // ps] = 1
        return m
    assert pins.check_page_mark(mark)


def _e4m3_mutant(kind):
    from oracle.fp8 import e4m3_decode

    def decode(codes):
        c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
        if kind == "bias_8":
            e = (c >> 3) & 0xF
            m = (c & 7) / 8.0
            v = np.where(e == 0, m * 2.0 ** -7, (1 + m) * np.exp2(e - 8.0))
            return np.where(c & 0x80, -v, v)
        if kind == "no_subnormals":
            v = e4m3_decode(codes)
            return np.where(((c >> 3) & 0xF) == 0, 0.0, v)
        return e4m3_decode(codes)
    return decode


@pytest.mark.parametrize("kind", ["bias_8", "no_subnormals"])
def test_e4m3_mutant_is_caught(kind):
    assert pins.check_e4m3_decode(_e4m3_mutant(kind))


def test_fp8_scale_mutant_is_caught():
    """Page scale indexed by slot instead of slot // page_size."""
    from oracle.fp8 import e4m3_decode
    from oracle import sparse_prefill

    def fn(q, k8, v8, ksc, vsc, ps, idx, tl, scale):
        def deq(c, sc):
            per = np.asarray(sc)[np.minimum(np.arange(c.shape[0]), sc.shape[0] - 1)]
            return e4m3_decode(c) * per[:, :, None]
        return sparse_prefill(q, deq(k8, ksc), deq(v8, vsc), idx, tl, scale)
    assert pins.check_fp8_attention(fn)
