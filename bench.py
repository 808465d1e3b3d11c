"""Benchmark: top-k sparse attention prefill on GB300 through the C ABI.

Default workload: the group-6 prefill chunk -- 8192 query rows at the end of a 32768-token
context, 6 query heads over 1 KV head, head_dim 256, topk 2051 uniformly drawn causal slots,
bf16 q/k/v ~ N(0, 1), seeded synthetic data.  One step = one qsa_sparse_prefill call over the
whole chunk (all stages of the hot path).

Timing: W untimed warm-up steps, then K steps each bracketed by CUDA events on the launching
stream; L2 is flushed (a 512 MiB memset) before every timed step, outside the events; the K
steps are bracketed by a barrier + synchronize; the max over ranks is reported.  SM clocks and
throttle reasons are sampled with nvidia-smi during the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--union G]
  python bench.py --impl reference ...     (the CPU oracle, timed on the host cores)

Under torchrun (N > 1) every rank runs its own full workload on its own GPU (weak scaling,
no collective on the data path); value = rows of all ranks / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse prefill query-rows/s (topk 2051, d=256, bf16) and % of gather/MMA roofline"
UNIT = "query-rows/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
_COMMON_KERNEL_SOURCES = ["top_sparse_attention_row_gb300/csrc/ptx.cuh",
                          "top_sparse_attention_row_gb300/csrc/internal.h",
                          "top_sparse_attention_row_gb300/csrc/paged.cuh",
                          "top_sparse_attention_row_gb300/csrc/compact.cuh"]
KERNEL_SOURCES = ["top_sparse_attention_row_gb300/csrc/prefill.cu"] + _COMMON_KERNEL_SOURCES
MLA_KERNEL_SOURCES = ["top_sparse_attention_row_gb300/csrc/mla.cu"] + _COMMON_KERNEL_SOURCES

DESCRIPTIONS = {
    "group6_32k": "group-6 prefill chunk: 8192 rows at the end of a 32768 context, 6 Q / 1 KV, "
                  "head_dim 256, topk 2051 uniform causal slots",
    "group12_128k": "group-12 long context: 8192 rows at the end of a 131072 context, 24 Q / 2 KV, "
                    "head_dim 256, topk 2051 uniform causal slots",
    "group12_128k_12q1kv": "group-12 long context, 12 Q / 1 KV rank shape",
    "union_8k": "8192-token prefill from position 0, 8 Q / 1 KV, topk 2048, random-walk indices",
    "mixed_paged": "mixed batch 512/2048/4096/8192 new tokens over prefixes 0/16k/32k/64k, "
                   "6 Q / 1 KV, topk 2051, per-row topk_len, paged cache (64), shuffled pages",
    "tiny": "tiny: 256 rows at positions 256..511, 6 Q / 1 KV, topk 128",
    "mla_8k": "MLA shape: 8192-token prefill from position 0, 8 heads, d_qk 576 (512 latent + 64 "
              "rope) / d_v 512 over one latent KV row per token, topk 2048, random-walk indices",
    "mla_4k": "MLA shape, 4096-token prefill (as mla_8k)",
    "mla_2k": "MLA shape, 2048-token prefill (as mla_8k; every row selects its whole prefix)",
}


def kernel_sha(mla: bool = False) -> str:
    h = hashlib.sha256()
    for rel in (MLA_KERNEL_SOURCES if mla else KERNEL_SOURCES):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_stats(w):
    """Algorithmic FLOPs / bytes of one call (unpadded heads, valid slots only)."""
    v = w.valid_counts().astype(np.int64)
    D, Hq, Hkv = w.head_dim, w.n_qheads, w.n_kvheads
    if w.meta.get("mla"):
        return mla_stats(w, v)
    elem = 1 if w.meta.get("fp8") else 2                     # cache bytes per element
    flops = int(4 * Hq * D * v.sum())                       # QK^T + PV, 2 flops per MAC
    idx = w.indices
    mask = idx >= 0
    if w.topk_len is not None:
        mask &= np.arange(idx.shape[1])[None, :] < np.clip(w.topk_len, 0, idx.shape[1])[:, None]
    unique_slots = int(np.unique(idx[mask]).size)
    kv_unique = unique_slots * Hkv * D * elem * 2            # K and V rows
    io = (2 * w.n_rows * Hq * D * 2 + idx.size * 4 + w.n_rows * Hq * 4
          + (0 if w.topk_len is None else w.n_rows * 4))
    gathered = int(v.sum()) * Hkv * D * elem * 2              # every (row, slot) K+V read
    return dict(flops=flops, bytes=kv_unique + io, unique_slots=unique_slots, gathered=gathered,
                valid_slots=int(v.sum()))


def mla_stats(w, v):
    """MLA shape: QK^T over 576 dims and PV over 512 per (row, head, valid slot); each slot is one
    1152-byte latent row, gathered once for both."""
    Dqk, Dv, H = w.q.shape[2], w.meta["d_v"], w.n_qheads
    flops = int(2 * H * (Dqk + Dv) * v.sum())
    idx = w.indices
    mask = idx >= 0
    if w.topk_len is not None:
        mask &= np.arange(idx.shape[1])[None, :] < np.clip(w.topk_len, 0, idx.shape[1])[:, None]
    unique_slots = int(np.unique(idx[mask]).size)
    io = (w.n_rows * H * (Dqk + Dv) * 2 + idx.size * 4 + w.n_rows * H * 4
          + (0 if w.topk_len is None else w.n_rows * 4))
    return dict(flops=flops, bytes=unique_slots * Dqk * 2 + io, unique_slots=unique_slots,
                gathered=int(v.sum()) * Dqk * 2, valid_slots=int(v.sum()))


# ------------------------------------------------------------------------- CPU oracle leg

_W = None


def _oracle_init(name, seed_kw, fp8_page_size=0):
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    global _W
    from top_sparse_attention_row_gb300 import workloads as W
    _W = W.make(name, **seed_kw)
    if fp8_page_size:
        _W = W.with_fp8_cache(_W, fp8_page_size)


def _oracle_rows(rows):
    import oracle
    w = _W
    if w.meta.get("mla"):
        oracle.sparse_mla_prefill_rows(w.q, w.k.reshape(w.k.shape[0], -1), w.indices, w.topk_len,
                                       w.scale, rows, w.meta["d_v"])
    elif w.meta.get("fp8"):
        m = w.meta
        oracle.sparse_prefill_fp8_rows(w.q, m["k8"], m["v8"], m["k_scale"], m["v_scale"],
                                       m["fp8_page_size"], w.indices, w.topk_len, w.scale, rows)
    else:
        oracle.sparse_prefill_rows(w.q, w.k, w.v, w.indices, w.topk_len, w.scale, rows)
    return len(rows)


def oracle_pool(name, seed_kw, cores, fp8_page_size=0):
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    ctx = mp.get_context("spawn")
    return ctx.Pool(cores, initializer=_oracle_init, initargs=(name, seed_kw, fp8_page_size))


def time_oracle(pool, n_rows, sample_rows, cores):
    rows = np.linspace(0, n_rows - 1, num=min(sample_rows, n_rows)).astype(np.int64)
    chunks = [c for c in np.array_split(rows, cores * 4) if len(c)]
    t0 = time.perf_counter()
    done = sum(pool.map(_oracle_rows, chunks))
    dt = time.perf_counter() - t0
    return done / dt, done, dt


# ------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------------- GPU leg

def max_over_ranks(values, device):
    """Element-wise max of per-rank timings (any torch.distributed backend)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def config_of(name, w, stats, union, paged, fp8, fp8_page_size, world):
    """The workload description shared, key for key, by the GPU arm and the reference arm."""
    return {"workload": DESCRIPTIONS.get(name, name), "name": name,
            "rows": w.n_rows, "n_qheads": w.n_qheads, "n_kvheads": w.n_kvheads,
            "head_dim": int(w.q.shape[2]), "topk": w.topk, "union_g": union,
            "valid_slots": stats["valid_slots"],
            "indices": ("logical positions + page table, translated in the kernels "
                        "(qsa_sparse_prefill_paged)" if paged else "physical slots"),
            "kv_cache": (f"e4m3 with fp32 scales per {fp8_page_size}-slot page and KV head, "
                         "dequantised in the gather (qsa_sparse_prefill_fp8)" if fp8 else "bf16"),
            "l2": "flushed before every timed GPU step (512 MiB memset outside the events)",
            "parallelism": f"{world} independent shard(s), no collective"}


class Prepared:
    """One workload's inputs on the host (pinned) and the device, and the library call."""

    def __init__(self, binding, W, name, *, fp8=False, paged=False, union=0, dev, seed_kw=None,
                 fp8_page_size=64, stream):
        import torch
        w = W.make(name, **(seed_kw or {}))
        if fp8:
            if w.meta.get("mla") or paged:
                raise SystemExit("--fp8 applies to the plain d=256 workloads")
            w = W.with_fp8_cache(w, fp8_page_size)
        self.w, self.name, self.fp8, self.paged, self.union = w, name, fp8, paged, union
        self.mla = bool(w.meta.get("mla"))
        if self.mla and paged:
            raise SystemExit("--paged applies to the d=256 workloads")
        if paged and "page_table" not in w.meta:
            raise SystemExit(f"--paged needs a paged workload; {name} has no page table")
        self.stats = workload_stats(w)
        self.binding, self.stream = binding, stream

        def bf(bits):
            return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)

        self.h_q = bf(w.q).pin_memory()
        if self.mla:   # one latent cache [S, 576]; V is its first 512 dims, not a separate tensor
            self.h_k = bf(w.k.reshape(w.k.shape[0], -1)).pin_memory()
            self.h_v = self.h_k[:0]
        elif fp8:   # e4m3 caches; their page scales travel with the metadata below
            self.h_k = torch.from_numpy(w.meta["k8"]).pin_memory()
            self.h_v = torch.from_numpy(w.meta["v8"]).pin_memory()
        else:
            self.h_k, self.h_v = bf(w.k).pin_memory(), bf(w.v).pin_memory()
        self.h_idx = torch.from_numpy(w.meta["logical_indices"] if paged else w.indices).pin_memory()
        self.h_tl = None if w.topk_len is None else torch.from_numpy(w.topk_len).pin_memory()
        self.h_meta = ()
        if fp8:
            self.h_meta = tuple(torch.from_numpy(np.ascontiguousarray(w.meta[k], dtype=np.float32))
                                .pin_memory() for k in ("k_scale", "v_scale"))
        if paged:   # ragged row offsets, per-request KV lengths and the page table
            self.h_meta = tuple(torch.from_numpy(np.ascontiguousarray(w.meta[k], dtype=np.int32))
                                .pin_memory() for k in ("cu_seqlens_q", "kv_lens_array", "page_table"))
        self.host_in = (self.h_q, self.h_k, self.h_v, self.h_idx, self.h_tl) + self.h_meta
        self.dev_in = tuple(None if t is None else t.to(dev) for t in self.host_in)
        q = self.dev_in[0]
        self.out = (torch.empty((w.n_rows, w.n_qheads, w.meta["d_v"]), dtype=torch.bfloat16, device=dev)
                    if self.mla else torch.empty_like(q))
        self.lse = torch.empty((w.n_rows, w.n_qheads), dtype=torch.float32, device=dev)
        self.ws = None
        self.forced = None   # forced geometry fields for the plain entry (None = selector)
        if union > 1 and not (self.mla or fp8 or paged):
            nb = binding.union_workspace_bytes(w.n_rows, w.topk, union)
            self.ws = torch.empty(max(nb, 256), dtype=torch.uint8, device=dev)
        if self.mla:
            self.geo = binding.select_mla_geometry(w.n_qheads, union, w.topk, w.n_rows)
        else:
            self.geo = binding.select_geometry(w.n_qheads, w.n_kvheads, union, w.topk, w.head_dim,
                                               w.n_rows)

    def call_on(self, dev_in, out, lse, ws):
        b, w, u, st = self.binding, self.w, self.union, self.stream
        q, k, v, idx, tl = dev_in[:5]
        meta = dev_in[5:]
        if self.mla:
            b.sparse_mla_prefill(q, k, idx, tl, w.scale, out=out, lse=lse, union_g=u, stream=st)
        elif self.fp8:
            ks, vs = meta
            b.sparse_prefill_fp8(q, k, v, ks, vs, w.meta["fp8_page_size"], idx, tl, w.scale, out=out,
                                 lse=lse, union_g=u, stream=st)
        elif self.paged:
            cu, kvl, pt = meta
            b.sparse_prefill_paged(q, k, v, idx, tl, cu, kvl, pt, w.meta["page_size"], w.scale,
                                   n_pages=w.meta["n_pages"], out=out, lse=lse, union_g=u, stream=st)
        else:
            b.sparse_prefill(q, k, v, idx, tl, w.scale, out=out, lse=lse, union_g=u, workspace=ws,
                             forced=self.forced, stream=st)

    def call(self):
        self.call_on(self.dev_in, self.out, self.lse, self.ws)

    def issued_mma_flops(self):
        """FLOPs the tensor cores execute, head padding included: every 128-slot tile of a work
        item runs QK^T (K = d_qk) and P.V (d_v output dims) at N = the padded query columns.
        Union tiles follow the union lists' lengths, read back from a union build."""
        import torch
        w, g = self.w, self.geo
        np_, chunks = g["n_pad"], g["head_chunks"]
        d_qk = int(w.q.shape[2])
        d_v = w.meta["d_v"] if self.mla else d_qk
        per_tile = 2 * 128 * np_ * (d_qk + d_v)
        if g["union_g"] > 1:
            phys = torch.from_numpy(np.ascontiguousarray(w.indices, dtype=np.int32)).to(self.out.device)
            _, _, _, ulen = self.binding.union_build(phys, self.dev_in[4], g["union_g"],
                                                     want_sorted=False)
            tiles = int(((ulen.cpu().numpy().astype(np.int64) + 127) // 128).sum())
        else:
            tiles = int(((w.valid_counts().astype(np.int64) + 127) // 128).sum())
        kv = 1 if self.mla else w.n_kvheads
        return tiles * kv * chunks * per_tile


def device_times(prep, steps, warmup, flush, stream):
    """W untimed calls, then `steps` calls each bracketed by CUDA events on the launching stream,
    with L2 flushed before each (outside the events) and ~0.5 ms of GPU spin after the flush so
    the host has enqueued the call before the start event runs."""
    import torch
    for _ in range(warmup):
        prep.call()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        torch.cuda._sleep(1 << 20)
        starts[i].record(stream)
        prep.call()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in zip(starts, ends)]


def roofline_of(prep, ms, peaks, peak_src, ceiling, issued):
    stats = prep.stats
    kernel_s = ms / 1e3
    t_tc = stats["flops"] / (peaks["bf16_tflops"] * 1e12)
    t_hbm = stats["bytes"] / (peaks["hbm_gbs"] * 1e9)
    bound = "tensor" if t_tc >= t_hbm else "hbm"
    if bound == "tensor":
        achieved, peak, unit = stats["flops"] / kernel_s / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    else:
        achieved, peak, unit = stats["bytes"] / kernel_s / 1e9, peaks["hbm_gbs"], "GB/s"
    r = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
         "peak_source": f"{peak_src} (MEASURED_PEAKS.json bf16 burst / hbm copy)",
         "algorithmic_flops": stats["flops"], "algorithmic_bytes": stats["bytes"],
         "roofline_us": max(t_tc, t_hbm) * 1e6,
         "issued_mma_flops": issued, "issued_tflops": issued / kernel_s / 1e12,
         "issued_frac": issued / kernel_s / 1e12 / peaks["bf16_tflops"],
         "gathered_bytes": stats["gathered"], "kernel_ms": ms}
    if ceiling and prep.union <= 1 and not prep.mla:
        r["gather_gbs"] = stats["gathered"] / kernel_s / 1e9
        r["gather_ceiling_gbs"] = ceiling
        r["frac_of_gather_ceiling"] = r["gather_gbs"] / ceiling
    return r


# workloads measured beside the headline one, each device-timed in its own launch configuration
SUB_CONFIGS = [
    ("tiny", {}), ("group12_128k", {}), ("group12_128k_12q1kv", {}),
    ("union_8k", {"union": 1}), ("union_8k", {"union": 2}), ("union_8k", {"union": 4}),
    ("mixed_paged", {"paged": True}), ("mla_8k", {"union": 0}), ("mla_8k", {"union": 2}),
    ("mla_8k", {"union": 4}), ("group6_32k", {"fp8": True}), ("union_8k", {"union": 4, "fp8": True}),
] + [(f"rows{r}_8k", {}) for r in (32, 64, 128, 256, 512, 1024)]   # query-count sweep


def run_gpu(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from top_sparse_attention_row_gb300 import binding, build as _build, workloads as W

    _build.build()
    binding.load_library()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    seed_kw = {} if world == 1 else {"seed": 1000 + rank}

    # CPU baseline pool (spawned, so safe whatever this process has done on the GPU).
    pool = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        pool = oracle_pool(args.config, seed_kw, cores, args.fp8_page_size if args.fp8 else 0)

    stream = torch.cuda.current_stream()
    prep = Prepared(binding, W, args.config, fp8=args.fp8, paged=args.paged, union=args.union,
                    dev=dev, seed_kw=seed_kw, fp8_page_size=args.fp8_page_size, stream=stream)
    w, stats, mla = prep.w, prep.stats, prep.mla
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)

    # gather ceiling on this workload's own K cache and selected rows (KV head 0), through a
    # view of the cache as 512-byte rows (for the 1152-byte MLA rows: the row holding each
    # selected slot's first bytes)
    k = prep.dev_in[1]
    valid = w.indices[w.indices >= 0].astype(np.int64)
    valid = valid * w.n_kvheads if not mla else (valid * w.q.shape[2]) // 256
    if args.fp8:   # 256-byte e4m3 rows: the 512-byte probe row holding each slot's row
        valid = valid // 2
    n_pieces = min(len(valid) // 128, 4096)
    table = torch.from_numpy(valid[: n_pieces * 128].astype(np.int32).reshape(n_pieces, 128)).to(dev)
    k_flat = k.reshape(-1)
    if k_flat.dtype != torch.bfloat16:   # e4m3 bytes: the probe reads 512-byte rows of the buffer
        k_flat = k_flat.view(torch.bfloat16)
    k_rows = k_flat[: (k_flat.numel() // 256) * 256].view(-1, 256)
    ceilings = {}
    for eng in ("tma", "cpasync"):
        binding.probe_gather_ceiling(k_rows, table, pieces_per_cta=200, engine=eng)
        ceilings[eng] = max(binding.probe_gather_ceiling(k_rows, table, engine=eng) for _ in range(3))
    ceiling_gbs = max(ceilings.values())

    for _ in range(args.warmup):
        prep.call()
    torch.cuda.synchronize()
    if binding.device_status(stream) != 0:
        raise RuntimeError("device wait timed out during warm-up")

    c0 = binding.counters()["kernel_launches"]
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    times = device_times(prep, args.steps, 0, flush, stream)
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - t_wall
    clocks = sampler.stop() if sampler else None
    launches = binding.counters()["kernel_launches"] - c0
    ms = sum(times) / len(times)
    if binding.device_status(stream) != 0:
        raise RuntimeError("device wait timed out during the timed region")

    # the pages' own regime: the same buffers every iteration, so L2 stays warm (median of 100)
    warm = []
    for _ in range(100):
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        prep.call()
        a1.record(stream)
        warm.append((a0, a1))
    torch.cuda.synchronize()
    warm_ms = statistics.median(x.elapsed_time(y) for x, y in warm)

    # end to end: pinned host inputs -> device, call, result -> host, every step
    e_out = torch.empty(prep.out.shape, dtype=prep.out.dtype).pin_memory()
    e_lse = torch.empty(prep.lse.shape, dtype=prep.lse.dtype).pin_memory()
    h2d_bytes = sum(t.numel() * t.element_size() for t in prep.host_in if t is not None)
    d2h = e_out.numel() * e_out.element_size() + e_lse.numel() * e_lse.element_size()

    # (1) serial: each step copies its inputs in, calls and copies O / LSE out on one stream,
    # nothing overlapped (the per-call latency a caller sees)
    def serial_step():
        for d, h in zip(prep.dev_in, prep.host_in):
            if d is not None:
                d.copy_(h, non_blocking=True)
        prep.call()
        e_out.copy_(prep.out, non_blocking=True)
        e_lse.copy_(prep.lse, non_blocking=True)

    serial_step()
    torch.cuda.synchronize()
    s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s_ev.record(stream)
    for _ in range(args.steps):
        serial_step()
    e_ev.record(stream)
    torch.cuda.synchronize()
    serial_ms = s_ev.elapsed_time(e_ev) / args.steps

    # (2) pipelined: two device input sets; step i+1's input copies and step i-1's output
    # copies run on their own streams while step i computes (every step still copies all of its
    # inputs in and its O / LSE out inside the timed region)
    sets = [prep.dev_in, tuple(None if t is None else torch.empty_like(t) for t in prep.dev_in)]
    outs = [(prep.out, prep.lse), (torch.empty_like(prep.out), torch.empty_like(prep.lse))]
    wss = [prep.ws, None if prep.ws is None else torch.empty_like(prep.ws)]
    copy_stream = torch.cuda.Stream(device=dev)
    out_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    read = [torch.cuda.Event(), torch.cuda.Event()]
    read_used = [False, False]

    def h2d(si):
        with torch.cuda.stream(copy_stream):
            for d, h in zip(sets[si], prep.host_in):
                if d is not None:
                    d.copy_(h, non_blocking=True)
            copied[si].record(copy_stream)

    def compute(si):
        stream.wait_event(copied[si])
        if read_used[si]:
            stream.wait_event(read[si])     # outs[si] is free once its copy-out has finished
        oo, ll = outs[si]
        prep.call_on(sets[si], oo, ll, wss[si])
        done[si].record(stream)
        out_stream.wait_event(done[si])
        with torch.cuda.stream(out_stream):
            e_out.copy_(oo, non_blocking=True)
            e_lse.copy_(ll, non_blocking=True)
            read[si].record(out_stream)
        read_used[si] = True

    def e2e_run(n):
        h2d(0)
        for i in range(n):
            if i + 1 < n:
                # set (i+1) % 2 is free once the kernel of step i-1 has consumed it
                if i >= 1:
                    copy_stream.wait_event(done[(i + 1) % 2])
                h2d((i + 1) % 2)
            compute(i % 2)

    e2e_run(3)
    torch.cuda.synchronize()
    flush.zero_()
    torch.cuda.synchronize()
    s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s_ev.record(stream)
    copy_stream.wait_event(s_ev)
    out_stream.wait_event(s_ev)
    e2e_run(args.steps)
    stream.wait_stream(copy_stream)
    stream.wait_stream(out_stream)
    e_ev.record(stream)
    torch.cuda.synchronize()
    e_ms = s_ev.elapsed_time(e_ev) / args.steps

    # max over ranks
    if world > 1:
        ms, e_ms, serial_ms = max_over_ranks([ms, e_ms, serial_ms], dev)

    if rank != 0:
        return None

    cpu = None
    if pool is not None:
        cores = os.cpu_count() or 1
        rps, n_done, dt = time_oracle(pool, w.n_rows, args.cpu_rows, cores)
        pool.close()
        pool.join()
        cpu = {"value": rps, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{n_done} of {w.n_rows} rows of the same workload (evenly spaced), "
                         f"numpy float64 oracle in {cores} spawned single-threaded processes, "
                         f"{dt:.2f} s wall"}

    peaks, peak_src = load_peaks()
    roofline = roofline_of(prep, ms, peaks, peak_src, ceiling_gbs, prep.issued_mma_flops())
    roofline["gather_ceiling_gbs"] = ceiling_gbs
    roofline["gather_ceiling_by_engine_gbs"] = ceilings
    roofline["gather_ceiling_source"] = ("qsa_probe_gather_ceiling on this workload's K cache and "
                                         "rows (the kernel's ring and engines, no compute; the "
                                         "faster engine)")
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        with open(tpath) as f:
            tj = json.load(f)
        key = (f"{args.config}:union{args.union}" + (":paged" if args.paged else "")
               + (":fp8" if args.fp8 else ""))
        ent = tj.get(key)
        if ent and ent.get("kernel_sha") == kernel_sha(mla):
            traffic = ent.get("dram_bytes_per_launch")
    roofline["traffic"] = traffic
    rows_total = w.n_rows * world
    line = {
        "metric": METRIC, "value": rows_total / (ms / 1e3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 MMA on e4m3 KV" if args.fp8 else "bf16",
        "data": "synthetic (seeded; no dataset or weights)",
        "config": config_of(args.config, w, stats, args.union, args.paged, args.fp8,
                            args.fp8_page_size, world),
        "geometry": prep.geo,
        "roofline": roofline,
        "e2e": {"value": rows_total / (e_ms / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
                "method": "public API per step: pinned-host inputs copied in, call, O and LSE "
                          "copied out; step i+1's input copies and step i-1's output copies "
                          "overlap step i on their own streams (two device buffer sets); no L2 "
                          "flush between steps (each step's copies replace the inputs)",
                "serial_ms_per_step": serial_ms,
                "serial_value": rows_total / (serial_ms / 1e3),
                "serial_method": "the same copies and call with nothing overlapped: copy in, "
                                 "call, copy out, one step after another on one stream"},
        "warm_l2": {"ms_per_step": warm_ms, "value": rows_total / (warm_ms / 1e3), "unit": UNIT,
                    "method": "median of 100 back-to-back calls on the same buffers (L2 warm), "
                              "the pages' timing regime; value above flushes L2 before each step"},
        "gpu_launches": launches,
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if world == 1 and not args.no_configs and args.config == "group6_32k" and not (
            args.fp8 or args.paged or args.union):
        del prep, sets, outs, wss
        torch.cuda.empty_cache()
        line["configs"] = run_sub_configs(binding, W, dev, stream, flush, peaks, peak_src,
                                          ceiling_gbs, args)
    return line


def run_sub_configs(binding, W, dev, stream, flush, peaks, peak_src, ceiling_gbs, args):
    """Every other workload, device-timed in this run as the headline one is (L2 flushed before
    each step); one record per workload and mode."""
    import torch
    recs = {}
    steps = max(3, min(args.steps, 10))
    for name, kw in SUB_CONFIGS:
        prep = Prepared(binding, W, name, fp8=kw.get("fp8", False), paged=kw.get("paged", False),
                        union=kw.get("union", 0), dev=dev, stream=stream)
        key = (name + (f" G={prep.union}" if "union" in kw else "") + (" paged" if prep.paged else "")
               + (" fp8" if prep.fp8 else ""))
        c0 = binding.counters()["kernel_launches"]
        sampler = ClockSampler(dev.index or 0)
        times = device_times(prep, steps, 3, flush, stream)
        clocks = sampler.stop()
        launches = (binding.counters()["kernel_launches"] - c0) // (steps + 3)
        if binding.device_status(stream) != 0:
            raise RuntimeError(f"device wait timed out on {key}")
        ms = sum(times) / len(times)
        roof = roofline_of(prep, ms, peaks, peak_src, None if prep.fp8 else ceiling_gbs,
                           prep.issued_mma_flops())
        recs[key] = {"ms": ms, "value": prep.w.n_rows / (ms / 1e3), "unit": UNIT,
                     "rows": prep.w.n_rows, "steps": steps,
                     "dtype": "f16 MMA on e4m3 KV" if prep.fp8 else "bf16",
                     "config": config_of(name, prep.w, prep.stats, prep.union, prep.paged, prep.fp8,
                                         64, 1),
                     "geometry": prep.geo, "roofline": roof, "clocks": clocks,
                     "launches_per_call": launches}
        if prep.geo.get("split", 1) > 1:
            # the same calls without the split (one CTA per row), for the sweep's comparison
            prep.forced = {"split": 1}
            t1 = device_times(prep, steps, 3, flush, stream)
            prep.forced = None
            ms1 = sum(t1) / len(t1)
            recs[key]["unsplit"] = {"ms": ms1, "value": prep.w.n_rows / (ms1 / 1e3)}
        del prep
        torch.cuda.empty_cache()
    return recs


def run_reference(args, rank, world):
    """The oracle as the reference arm, timed on this host's cores."""
    if rank != 0:
        return None
    from top_sparse_attention_row_gb300 import workloads as W
    w = W.make(args.config)
    if args.fp8:
        w = W.with_fp8_cache(w, args.fp8_page_size)
    stats = workload_stats(w)
    cores = os.cpu_count() or 1
    pool = oracle_pool(args.config, {}, cores, args.fp8_page_size if args.fp8 else 0)
    sample = min(w.n_rows, args.cpu_rows)
    for _ in range(args.warmup):
        time_oracle(pool, w.n_rows, max(cores, sample // 8), cores)
    vals = []
    for _ in range(args.steps):
        rps, _, _ = time_oracle(pool, w.n_rows, sample, cores)
        vals.append(rps)
    pool.close()
    pool.join()
    value = statistics.median(vals)
    ms = 1e3 * w.n_rows / value
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; no dataset or weights)",
        "impl": "reference",
        "config": config_of(args.config, w, stats, args.union, args.paged, args.fp8,
                            args.fp8_page_size, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{sample} of {w.n_rows} rows per step (evenly spaced), numpy "
                                   f"float64 oracle in {cores} spawned single-threaded processes"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_page_split(args):
    """The touched-page re-layout of a decode step (qsa_split_touched_pages: mark + masked split)
    on a 4096-page pool of 256-token pages, against the full split of the same pool.  Time per
    call with CUDA events; the L2 is flushed before every timed call."""
    import torch
    from top_sparse_attention_row_gb300 import binding, build as _build, workloads as W
    _build.build()
    binding.load_library()
    dev = torch.device("cuda", 0)
    w = W.make_page_split()
    n, sps, dps, secs = w["n_src_pages"], w["src_page_size"], w["dst_page_size"], w["section_bytes"]
    src = torch.from_numpy(w["pool"]).to(dev)
    dst = torch.empty_like(src)
    idx = torch.from_numpy(w["indices"]).to(dev)
    mark = torch.empty(n, dtype=torch.uint8, device=dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(args.steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    c0 = binding.counters()["kernel_launches"]
    sampler = ClockSampler(0)
    masked_ms = timed(lambda: binding.split_touched_pages(idx, src, dst, mark, n, sps, dps, secs,
                                                          stream=stream))
    clocks = sampler.stop()
    launches = (binding.counters()["kernel_launches"] - c0) // (args.steps + args.warmup)
    full_ms = timed(lambda: binding.page_split(src, dst, n, sps, dps, secs, stream=stream))
    touched = int(mark.sum().item())
    page_bytes = sps * sum(secs)
    useful = 2 * touched * page_bytes + idx.numel() * 4 + n          # touched pages r+w, indices, mark
    peaks, peak_src = load_peaks()
    hbm = peaks["hbm_gbs"]
    return {
        "metric": "touched-page split time per decode step", "value": masked_ms, "unit": "ms",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": masked_ms,
        "higher_is_better": False, "dtype": "u8", "data": "synthetic (seeded)",
        "config": {"workload": f"{n} pages of {sps} tokens x {sum(secs)} B ({secs}), split to pages of "
                               f"{dps}; 8 requests x 512-token windows", "name": "swa_page_split",
                   "touched_pages": touched, "l2": "flushed before every timed call"},
        "full_split_ms": full_ms,
        "roofline": {"bound": "hbm", "kernel": "page_split_kernel (full split)",
                     "achieved": 2 * n * page_bytes / (full_ms * 1e-3) / 1e9, "peak": hbm,
                     "unit": "GB/s", "frac": 2 * n * page_bytes / (full_ms * 1e-3) / 1e9 / hbm,
                     "peak_source": peak_src, "traffic": None},
        "masked_useful_gbs": useful / (masked_ms * 1e-3) / 1e9,
        "gpu_launches": launches, "clocks": clocks,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="group6_32k")
    ap.add_argument("--union", type=int, default=0)
    ap.add_argument("--paged", action="store_true",
                    help="paged workloads: pass logical positions and the page table "
                         "(qsa_sparse_prefill_paged) instead of translated slots")
    ap.add_argument("--fp8", action="store_true",
                    help="d=256 workloads: e4m3 K/V caches with per-page scales "
                         "(qsa_sparse_prefill_fp8)")
    ap.add_argument("--fp8-page-size", type=int, default=64)
    ap.add_argument("--cpu-rows", type=int, default=8192)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload records timed beside the default headline line")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if args.config == "swa_page_split":
        line = run_page_split(args) if rank == 0 else None
    else:
        line = run_gpu(args, rank, world, local_rank)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
