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
