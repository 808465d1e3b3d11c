"""Every-row oracle checks at full size, spread over the host cores (test plumbing).

The GPU results of a full-size call are written to .npy files; a pool of SPAWNED worker
processes (never forked: a process forked after CUDA initialisation can hang) regenerates the
same seeded workload, runs the float64 oracle on its share of the rows and compares them with
the GPU rows it reads back from those files.  Only per-row error figures travel back, so a
8192-row x 24-head call never has to hold the oracle's float64 output in one process.

The comparison bounds are those of ``helpers``: max |dO| <= 2e-2, |dLSE| <= 1e-3 * max(1, |LSE|),
and -inf LSE exactly where the oracle has it.  Failures name the worst row.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import tempfile

import numpy as np

from helpers import O_ATOL, LSE_RTOL

_CACHE = {}


def _workload(spec):
    """spec = (name, variant): variant "" (bf16 caches), "fp8:<page size>" (e4m3 caches)."""
    if spec not in _CACHE:
        from top_sparse_attention_row_gb300 import workloads as W
        name, variant = spec
        w = W.make(name)
        if variant.startswith("fp8:"):
            w = W.with_fp8_cache(w, int(variant.split(":")[1]))
        _CACHE.clear()               # one full-size workload per worker at a time
        _CACHE[spec] = w
    return _CACHE[spec]


def _oracle_rows(w, kind, rows):
    import oracle
    if kind == "mla":
        return oracle.sparse_mla_prefill_rows(w.q, w.k.reshape(w.k.shape[0], -1), w.indices,
                                              w.topk_len, w.scale, rows, w.meta["d_v"])
    if kind == "fp8":
        m = w.meta
        return oracle.sparse_prefill_fp8_rows(w.q, m["k8"], m["v8"], m["k_scale"], m["v_scale"],
                                              m["fp8_page_size"], w.indices, w.topk_len, w.scale,
                                              rows)
    if kind == "paged":
        m = w.meta
        return oracle.sparse_prefill_paged_rows(w.q, w.k, w.v, m["logical_indices"], w.topk_len,
                                                m["cu_seqlens_q"], m["kv_lens_array"],
                                                m["page_table"], m["page_size"], w.scale, rows,
                                                m["n_pages"])
    return oracle.sparse_prefill_rows(w.q, w.k, w.v, w.indices, w.topk_len, w.scale, rows)


def _bf16_bits_to_f64(bits):
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32).astype(np.float64)


def _compare_chunk(args):
    spec, kind, rows, out_path, lse_path = args
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    w = _workload(spec)
    O, L = _oracle_rows(w, kind, rows)
    out = np.load(out_path, mmap_mode="r")
    lse = np.load(lse_path, mmap_mode="r")
    o = _bf16_bits_to_f64(out[rows])
    l = np.asarray(lse[rows], dtype=np.float64)
    dO = np.abs(o - O).reshape(len(rows), -1).max(axis=1)
    inf_ref, inf_got = np.isneginf(L), np.isneginf(l)
    mism = (inf_ref != inf_got).sum(axis=1)
    fin = ~inf_ref & ~inf_got
    rel = np.where(fin, np.abs(np.where(fin, l, 0.0) - np.where(fin, L, 0.0))
                   / np.maximum(1.0, np.abs(np.where(fin, L, 0.0))), 0.0)
    return rows, dO, rel.max(axis=1), mism


def _union_chunk(args):
    spec, G, g0, g1, idx_path, bits_path, len_path = args
    import oracle
    w = _workload(spec)
    r0, r1 = g0 * G, min(g1 * G, w.n_rows)
    e_idx, e_bits, e_len = oracle.union_build(w.indices[r0:r1], None if w.topk_len is None
                                              else w.topk_len[r0:r1], G)
    uidx = np.load(idx_path, mmap_mode="r")[g0:g1]
    ubits = np.load(bits_path, mmap_mode="r")[g0:g1]
    ulen = np.load(len_path, mmap_mode="r")[g0:g1]
    bad = []
    for i in range(g1 - g0):
        if (ulen[i] != e_len[i] or not np.array_equal(uidx[i], e_idx[i])
                or not np.array_equal(ubits[i], e_bits[i])):
            bad.append(g0 + i)
    return bad


class OraclePool:
    def __init__(self, processes=None):
        for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        self.n = processes or os.cpu_count() or 1
        self.pool = mp.get_context("spawn").Pool(self.n)
        self.tmp = tempfile.TemporaryDirectory(prefix="qsa_oracle_")

    def close(self):
        self.pool.close()
        self.pool.join()
        self.tmp.cleanup()

    def _save(self, name, arr):
        path = os.path.join(self.tmp.name, name + ".npy")
        np.save(path, arr)
        return path

    def _chunks(self, n, parts):
        return [c for c in np.array_split(np.arange(n), parts) if len(c)]

    def check_all_rows(self, spec, kind, out, lse, what):
        """out (bf16 torch tensor [R, H, Dv]) and lse ([R, H] fp32) against the oracle on every
        row; asserts the bounds and returns (max |dO|, max rel |dLSE|)."""
        o = out.view(dtype=__import__("torch").int16).cpu().numpy().view(np.uint16)
        l = lse.float().cpu().numpy()
        po, pl = self._save("out", o), self._save("lse", l)
        R = o.shape[0]
        jobs = [(spec, kind, rows, po, pl) for rows in self._chunks(R, self.n * 4)]
        dO = np.zeros(R)
        dL = np.zeros(R)
        mism = np.zeros(R, dtype=np.int64)
        for rows, a, b, c in self.pool.imap_unordered(_compare_chunk, jobs):
            dO[rows], dL[rows], mism[rows] = a, b, c
        worst_o, worst_l = int(np.argmax(dO)), int(np.argmax(dL))
        assert mism.sum() == 0, (f"{what}: LSE -inf mismatches on {int((mism > 0).sum())} rows, "
                                 f"first row {int(np.flatnonzero(mism)[0])}")
        assert dO[worst_o] <= O_ATOL, f"{what}: max |dO| = {dO[worst_o]:.3e} at row {worst_o}"
        assert dL[worst_l] <= LSE_RTOL, (f"{what}: max rel |dLSE| = {dL[worst_l]:.3e} at row "
                                         f"{worst_l}")
        return float(dO[worst_o]), float(dL[worst_l])

    def check_union_build(self, spec, G, uidx, ubits, ulen, what):
        """The GPU's union lists, bits and lengths (numpy) equal the oracle's, group by group."""
        n_groups = uidx.shape[0]
        pi, pb, pn = self._save("uidx", uidx), self._save("ubits", ubits), self._save("ulen", ulen)
        bounds = np.linspace(0, n_groups, self.n * 4 + 1).astype(int)
        jobs = [(spec, G, int(a), int(b), pi, pb, pn) for a, b in zip(bounds[:-1], bounds[1:])
                if b > a]
        bad = sorted(g for part in self.pool.imap_unordered(_union_chunk, jobs) for g in part)
        assert not bad, f"{what}: {len(bad)} groups differ from the oracle, first group {bad[0]}"
