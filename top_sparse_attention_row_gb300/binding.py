"""Thin ctypes binding over libqsa.so (argument marshalling only).

Every step of the sparse prefill runs in the library's CUDA kernels; this module only
checks tensor dtypes / shapes / devices and passes raw pointers and sizes through the C ABI
declared in ``include/qsa.h``.  It raises ``RuntimeError`` on any non-OK status and refuses
to run when the library has not been built -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libqsa.so")

QSA_OK = 0
STATUS_NAMES = {0: "QSA_OK", 1: "QSA_ERR_INVALID_ARG", 2: "QSA_ERR_UNSUPPORTED",
                3: "QSA_ERR_WORKSPACE", 4: "QSA_ERR_CUDA", 5: "QSA_ERR_TIMEOUT"}

# Every symbol include/qsa.h declares (checked by the CPU test suite).
EXPORTED = ["qsa_sparse_prefill", "qsa_sparse_prefill_ex", "qsa_union_workspace_bytes",
            "qsa_workspace_bytes",
            "qsa_union_build", "qsa_select_geometry", "qsa_get_counters", "qsa_reset_counters",
            "qsa_status_string", "qsa_version", "qsa_get_device_status",
            "qsa_sparse_prefill_noalloc", "qsa_probe_gather_ceiling",
            "qsa_sparse_prefill_paged", "qsa_sparse_mla_prefill", "qsa_select_mla_geometry",
            "qsa_page_mark", "qsa_page_split", "qsa_split_touched_pages",
            "qsa_sparse_prefill_fp8", "qsa_debug_stall_next_call", "qsa_sparse_mla_prefill_paged",
            "qsa_sparse_prefill_fp8_paged"]

# Size of the library-owned scratch array used by qsa_sparse_prefill_noalloc (include/qsa.h).
NOALLOC_SCRATCH_BYTES = 32 << 20


class Geometry(ctypes.Structure):
    _fields_ = [("tile_tokens", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("n_pad", ctypes.c_int32), ("cols", ctypes.c_int32),
                ("head_chunks", ctypes.c_int32), ("union_g", ctypes.c_int32),
                ("grid", ctypes.c_int32), ("threads", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("tmem_cols", ctypes.c_int32),
                ("n_items", ctypes.c_int64), ("split", ctypes.c_int32)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class Counters(ctypes.Structure):
    _fields_ = [("calls_per_token", ctypes.c_uint64), ("calls_union", ctypes.c_uint64),
                ("union_fallbacks", ctypes.c_uint64), ("step_downs", ctypes.c_uint64),
                ("kernel_launches", ctypes.c_uint64)]

    def as_dict(self):
        return {name: int(getattr(self, name)) for name, _ in self._fields_}


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libqsa.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libqsa.so not built at {path}; run __graft_entry__.build() "
                           "or python -m top_sparse_attention_row_gb300.build")
    lib = ctypes.CDLL(path)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.qsa_sparse_prefill.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, f32, i32, vp]
    lib.qsa_sparse_prefill.restype = ctypes.c_int
    lib.qsa_sparse_prefill_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, f32, i32,
                                          i64, vp, sz, ctypes.POINTER(Geometry), vp]
    lib.qsa_sparse_prefill_ex.restype = ctypes.c_int
    lib.qsa_sparse_prefill_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, f32,
                                               i32, vp]
    lib.qsa_sparse_prefill_noalloc.restype = ctypes.c_int
    lib.qsa_sparse_prefill_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i32, i32,
                                             i32, i64, i32, i32, i32, i32, f32, i32, vp]
    lib.qsa_sparse_prefill_paged.restype = ctypes.c_int
    lib.qsa_sparse_mla_prefill.argtypes = [vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, f32, i32,
                                           i64, vp]
    lib.qsa_sparse_mla_prefill.restype = ctypes.c_int
    lib.qsa_select_mla_geometry.argtypes = [i32, i32, i32, i32, i32, i64, i32, ctypes.POINTER(Geometry)]
    lib.qsa_select_mla_geometry.restype = ctypes.c_int
    lib.qsa_page_mark.argtypes = [vp, i64, i32, i64, vp, vp]
    lib.qsa_page_mark.restype = ctypes.c_int
    lib.qsa_page_split.argtypes = [vp, vp, vp, i64, i32, i32, i32, vp, vp]
    lib.qsa_page_split.restype = ctypes.c_int
    lib.qsa_split_touched_pages.argtypes = [vp, i64, vp, vp, vp, i64, i32, i32, i32, vp, vp]
    lib.qsa_split_touched_pages.restype = ctypes.c_int
    lib.qsa_sparse_prefill_fp8.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, i64, i32, i32,
                                           i32, i32, f32, i32, i64, vp]
    lib.qsa_sparse_prefill_fp8.restype = ctypes.c_int
    lib.qsa_sparse_prefill_fp8_paged.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp,
                                                 i64, i32, i32, i32, i64, i32, i32, i32, i32, f32,
                                                 i32, vp]
    lib.qsa_sparse_prefill_fp8_paged.restype = ctypes.c_int
    lib.qsa_debug_stall_next_call.argtypes = []
    lib.qsa_debug_stall_next_call.restype = None
    lib.qsa_sparse_mla_prefill_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i32, i32,
                                                 i32, i64, i32, i32, i32, i32, f32, i32, vp]
    lib.qsa_sparse_mla_prefill_paged.restype = ctypes.c_int
    lib.qsa_probe_gather_ceiling.argtypes = [vp, i64, vp, i64, i32, i32, ctypes.POINTER(f32), vp]
    lib.qsa_probe_gather_ceiling.restype = ctypes.c_int
    for name in ("qsa_union_workspace_bytes", "qsa_workspace_bytes"):
        getattr(lib, name).argtypes = [i64, i32, i32]
        getattr(lib, name).restype = sz
    lib.qsa_union_build.argtypes = [vp, vp, i64, i32, i32, i64, vp, vp, vp, vp, vp]
    lib.qsa_union_build.restype = ctypes.c_int
    lib.qsa_select_geometry.argtypes = [i32, i32, i32, i32, i32, i64, i32, ctypes.POINTER(Geometry)]
    lib.qsa_select_geometry.restype = ctypes.c_int
    lib.qsa_get_counters.argtypes = [ctypes.POINTER(Counters)]
    lib.qsa_get_counters.restype = None
    lib.qsa_reset_counters.argtypes = []
    lib.qsa_reset_counters.restype = None
    lib.qsa_status_string.argtypes = [ctypes.c_int]
    lib.qsa_status_string.restype = ctypes.c_char_p
    lib.qsa_version.argtypes = []
    lib.qsa_version.restype = ctypes.c_char_p
    lib.qsa_get_device_status.argtypes = [vp, ctypes.POINTER(i32)]
    lib.qsa_get_device_status.restype = ctypes.c_int
    _lib = lib
    return lib


def _check(status: int, what: str):
    if status != QSA_OK:
        msg = load_library().qsa_status_string(status).decode()
        raise RuntimeError(f"{what} failed: {STATUS_NAMES.get(status, status)} ({msg})")


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _require(t, dtype, name, ndim=None):
    import torch
    if t is None:
        return
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")


def sparse_prefill(q, k_cache, v_cache, indices, topk_len, scale: float, *, out=None, lse=None,
                   union_g: int = 0, n_kv_slots: int = 0, workspace=None, forced: Optional[dict] = None,
                   want_lse: bool = True, stream=None):
    """O (bf16 [R, Hq, D]) and LSE (fp32 [R, Hq]) of top-k sparse attention prefill.

    q [R, Hq, D] bf16, k_cache / v_cache [S, Hkv, D] bf16, indices [R, topk] int32 (physical
    slots, negative = padding), topk_len [R] int32 or None.  Calls qsa_sparse_prefill (or the
    _ex entry when n_kv_slots / workspace / forced are given) on the current stream.
    """
    import torch
    lib = load_library()
    _require(q, torch.bfloat16, "q", 3)
    _require(k_cache, torch.bfloat16, "k_cache", 3)
    _require(v_cache, torch.bfloat16, "v_cache", 3)
    _require(indices, torch.int32, "indices", 2)
    _require(topk_len, torch.int32, "topk_len", 1)
    R, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    topk = indices.shape[1]
    if indices.shape[0] != R or (topk_len is not None and topk_len.shape[0] != R):
        raise ValueError("indices / topk_len rows must match q")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((R, Hq), dtype=torch.float32, device=q.device)
    _require(out, torch.bfloat16, "out", 3)
    _require(lse, torch.float32, "lse", 2)
    s = _stream_ptr(stream)
    if n_kv_slots or workspace is not None or forced:
        g = None
        if forced:
            g = Geometry()
            for k, v in forced.items():
                setattr(g, k, v)
        ws_ptr = None if workspace is None else workspace.data_ptr()
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        st = lib.qsa_sparse_prefill_ex(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(indices),
                                       _ptr(topk_len), _ptr(out), _ptr(lse), R, Hq, Hkv, D, topk,
                                       float(scale), int(union_g), int(n_kv_slots), ws_ptr, ws_bytes,
                                       None if g is None else ctypes.byref(g), s)
    else:
        st = lib.qsa_sparse_prefill(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(indices),
                                    _ptr(topk_len), _ptr(out), _ptr(lse), R, Hq, Hkv, D, topk,
                                    float(scale), int(union_g), s)
    _check(st, "qsa_sparse_prefill")
    return out, lse


def sparse_prefill_paged(q, k_cache, v_cache, indices, topk_len, cu_seqlens_q, kv_lens, page_table,
                         page_size: int, scale: float, *, n_pages: int = 0, out=None, lse=None,
                         union_g: int = 0, want_lse: bool = True, stream=None):
    """Paged call (qsa_sparse_prefill_paged): indices [R, topk] int32 are logical positions in
    each row's request; cu_seqlens_q [n_requests + 1] int32 row offsets; kv_lens [n_requests]
    int32 or None; page_table [n_requests, pages_per_req] int32; k_cache / v_cache
    [n_pages * page_size, Hkv, D] bf16.  The translation to physical slots runs in the kernels."""
    import torch
    lib = load_library()
    _require(q, torch.bfloat16, "q", 3)
    _require(k_cache, torch.bfloat16, "k_cache", 3)
    _require(v_cache, torch.bfloat16, "v_cache", 3)
    _require(indices, torch.int32, "indices", 2)
    _require(topk_len, torch.int32, "topk_len", 1)
    _require(cu_seqlens_q, torch.int32, "cu_seqlens_q", 1)
    _require(kv_lens, torch.int32, "kv_lens", 1)
    _require(page_table, torch.int32, "page_table", 2)
    R, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    topk = indices.shape[1]
    n_req = page_table.shape[0]
    if indices.shape[0] != R or (topk_len is not None and topk_len.shape[0] != R):
        raise ValueError("indices / topk_len rows must match q")
    if cu_seqlens_q.shape[0] != n_req + 1 or (kv_lens is not None and kv_lens.shape[0] != n_req):
        raise ValueError("cu_seqlens_q / kv_lens must match the page table's requests")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((R, Hq), dtype=torch.float32, device=q.device)
    _require(out, torch.bfloat16, "out", 3)
    _require(lse, torch.float32, "lse", 2)
    st = lib.qsa_sparse_prefill_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(indices),
                                      _ptr(topk_len), _ptr(cu_seqlens_q), _ptr(kv_lens),
                                      _ptr(page_table), _ptr(out), _ptr(lse), R, n_req,
                                      page_table.shape[1], int(page_size), int(n_pages), Hq, Hkv,
                                      D, topk, float(scale), int(union_g), _stream_ptr(stream))
    _check(st, "qsa_sparse_prefill_paged")
    return out, lse


def sparse_prefill_fp8_paged(q, k_cache, v_cache, k_scale, v_scale, fp8_page_size: int, indices,
                             topk_len, cu_seqlens_q, kv_lens, page_table, page_size: int,
                             scale: float, *, n_pages: int = 0, out=None, lse=None,
                             union_g: int = 0, want_lse: bool = True, stream=None):
    """FP8 caches over a paged pool (qsa_sparse_prefill_fp8_paged): the e4m3 caches and scales of
    sparse_prefill_fp8 (scale granularity fp8_page_size) with the logical indices and page table
    of sparse_prefill_paged (pool page size page_size)."""
    import torch
    lib = load_library()
    _require(q, torch.bfloat16, "q", 3)
    _require(k_cache, torch.uint8, "k_cache", 3)
    _require(v_cache, torch.uint8, "v_cache", 3)
    _require(k_scale, torch.float32, "k_scale", 2)
    _require(v_scale, torch.float32, "v_scale", 2)
    _require(indices, torch.int32, "indices", 2)
    _require(topk_len, torch.int32, "topk_len", 1)
    _require(cu_seqlens_q, torch.int32, "cu_seqlens_q", 1)
    _require(kv_lens, torch.int32, "kv_lens", 1)
    _require(page_table, torch.int32, "page_table", 2)
    R, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    topk = indices.shape[1]
    n_req = page_table.shape[0]
    if indices.shape[0] != R or (topk_len is not None and topk_len.shape[0] != R):
        raise ValueError("indices / topk_len rows must match q")
    if cu_seqlens_q.shape[0] != n_req + 1 or (kv_lens is not None and kv_lens.shape[0] != n_req):
        raise ValueError("cu_seqlens_q / kv_lens must match the page table's requests")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((R, Hq), dtype=torch.float32, device=q.device)
    _require(out, torch.bfloat16, "out", 3)
    _require(lse, torch.float32, "lse", 2)
    st = lib.qsa_sparse_prefill_fp8_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                          _ptr(v_scale), int(fp8_page_size), _ptr(indices),
                                          _ptr(topk_len), _ptr(cu_seqlens_q), _ptr(kv_lens),
                                          _ptr(page_table), _ptr(out), _ptr(lse), R, n_req,
                                          page_table.shape[1], int(page_size), int(n_pages), Hq,
                                          Hkv, D, topk, float(scale), int(union_g),
                                          _stream_ptr(stream))
    _check(st, "qsa_sparse_prefill_fp8_paged")
    return out, lse


def sparse_prefill_fp8(q, k_cache, v_cache, k_scale, v_scale, page_size: int, indices, topk_len,
                       scale: float, *, out=None, lse=None, union_g: int = 0, n_kv_slots: int = 0,
                       want_lse: bool = True, stream=None):
    """FP8 caches (qsa_sparse_prefill_fp8): k_cache / v_cache [S, Hkv, D] uint8 e4m3 codes,
    k_scale / v_scale [ceil(S / page_size), Hkv] fp32; otherwise as sparse_prefill."""
    import torch
    lib = load_library()
    _require(q, torch.bfloat16, "q", 3)
    _require(k_cache, torch.uint8, "k_cache", 3)
    _require(v_cache, torch.uint8, "v_cache", 3)
    _require(k_scale, torch.float32, "k_scale", 2)
    _require(v_scale, torch.float32, "v_scale", 2)
    _require(indices, torch.int32, "indices", 2)
    _require(topk_len, torch.int32, "topk_len", 1)
    R, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    topk = indices.shape[1]
    if indices.shape[0] != R or (topk_len is not None and topk_len.shape[0] != R):
        raise ValueError("indices / topk_len rows must match q")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((R, Hq), dtype=torch.float32, device=q.device)
    _require(out, torch.bfloat16, "out", 3)
    _require(lse, torch.float32, "lse", 2)
    st = lib.qsa_sparse_prefill_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                    _ptr(v_scale), int(page_size), _ptr(indices), _ptr(topk_len),
                                    _ptr(out), _ptr(lse), R, Hq, Hkv, D, topk, float(scale),
                                    int(union_g), int(n_kv_slots), _stream_ptr(stream))
    _check(st, "qsa_sparse_prefill_fp8")
    return out, lse


def sparse_mla_prefill(q, kv_cache, indices, topk_len, scale: float, *, out=None, lse=None,
                       union_g: int = 0, n_kv_slots: int = 0, want_lse: bool = True, stream=None):
    """MLA shape (qsa_sparse_mla_prefill): q [R, H, 576] bf16, kv_cache [S, 576] bf16 (the first
    512 dims are the value), indices [R, topk] int32 physical slots, topk_len [R] int32 or None.
    Returns O [R, H, 512] bf16 and LSE [R, H] fp32."""
    import torch
    lib = load_library()
    _require(q, torch.bfloat16, "q", 3)
    _require(kv_cache, torch.bfloat16, "kv_cache", 2)
    _require(indices, torch.int32, "indices", 2)
    _require(topk_len, torch.int32, "topk_len", 1)
    R, H, Dqk = q.shape
    Dv = 512
    topk = indices.shape[1]
    if indices.shape[0] != R or (topk_len is not None and topk_len.shape[0] != R):
        raise ValueError("indices / topk_len rows must match q")
    if kv_cache.shape[1] != Dqk:
        raise ValueError("kv_cache rows must have q's head dim")
    if out is None:
        out = torch.empty((R, H, Dv), dtype=torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((R, H), dtype=torch.float32, device=q.device)
    _require(out, torch.bfloat16, "out", 3)
    _require(lse, torch.float32, "lse", 2)
    st = lib.qsa_sparse_mla_prefill(_ptr(q), _ptr(kv_cache), _ptr(indices), _ptr(topk_len), _ptr(out),
                                    _ptr(lse), R, H, Dqk, Dv, topk, float(scale), int(union_g),
                                    int(n_kv_slots), _stream_ptr(stream))
    _check(st, "qsa_sparse_mla_prefill")
    return out, lse


def sparse_mla_prefill_paged(q, kv_cache, indices, topk_len, cu_seqlens_q, kv_lens, page_table,
                             page_size: int, scale: float, *, n_pages: int = 0, out=None, lse=None,
                             union_g: int = 0, want_lse: bool = True, stream=None):
    """MLA shape over a paged latent cache (qsa_sparse_mla_prefill_paged): logical indices,
    ragged row offsets and a page table as in sparse_prefill_paged."""
    import torch
    lib = load_library()
    _require(q, torch.bfloat16, "q", 3)
    _require(kv_cache, torch.bfloat16, "kv_cache", 2)
    _require(indices, torch.int32, "indices", 2)
    _require(topk_len, torch.int32, "topk_len", 1)
    _require(cu_seqlens_q, torch.int32, "cu_seqlens_q", 1)
    _require(kv_lens, torch.int32, "kv_lens", 1)
    _require(page_table, torch.int32, "page_table", 2)
    R, H, Dqk = q.shape
    n_req = page_table.shape[0]
    if cu_seqlens_q.shape[0] != n_req + 1 or (kv_lens is not None and kv_lens.shape[0] != n_req):
        raise ValueError("cu_seqlens_q / kv_lens must match the page table's requests")
    if out is None:
        out = torch.empty((R, H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((R, H), dtype=torch.float32, device=q.device)
    st = lib.qsa_sparse_mla_prefill_paged(_ptr(q), _ptr(kv_cache), _ptr(indices), _ptr(topk_len),
                                          _ptr(cu_seqlens_q), _ptr(kv_lens), _ptr(page_table),
                                          _ptr(out), _ptr(lse), R, n_req, page_table.shape[1],
                                          int(page_size), int(n_pages), H, Dqk, 512,
                                          indices.shape[1], float(scale), int(union_g),
                                          _stream_ptr(stream))
    _check(st, "qsa_sparse_mla_prefill_paged")
    return out, lse


def select_mla_geometry(n_heads, union_g, topk, n_rows, num_sms=0, d_qk=576, d_v=512) -> dict:
    g = Geometry()
    st = load_library().qsa_select_mla_geometry(n_heads, union_g, topk, d_qk, d_v, n_rows, num_sms,
                                                ctypes.byref(g))
    _check(st, "qsa_select_mla_geometry")
    return g.as_dict()


def _sections(section_bytes):
    arr = (ctypes.c_int32 * len(section_bytes))(*[int(b) for b in section_bytes])
    return arr, len(section_bytes)


def page_mark(indices, src_page_size: int, n_src_pages: int, *, mark=None, stream=None):
    """qsa_page_mark: uint8 [n_src_pages] (zeroed, then 1 on every page a valid index touches)."""
    import torch
    _require(indices, torch.int32, "indices", None)
    if mark is None:
        mark = torch.empty(n_src_pages, dtype=torch.uint8, device=indices.device)
    st = load_library().qsa_page_mark(_ptr(indices), indices.numel(), int(src_page_size),
                                      int(n_src_pages), _ptr(mark), _stream_ptr(stream))
    _check(st, "qsa_page_mark")
    return mark


def page_split(src_pool, dst_pool, n_src_pages: int, src_page_size: int, dst_page_size: int,
               section_bytes, *, mark=None, stream=None):
    """qsa_page_split over flat uint8 pools; mark None = every page."""
    arr, n = _sections(section_bytes)
    st = load_library().qsa_page_split(_ptr(src_pool), _ptr(dst_pool), _ptr(mark), int(n_src_pages),
                                       int(src_page_size), int(dst_page_size), n, arr,
                                       _stream_ptr(stream))
    _check(st, "qsa_page_split")
    return dst_pool


def split_touched_pages(indices, src_pool, dst_pool, mark, n_src_pages: int, src_page_size: int,
                        dst_page_size: int, section_bytes, *, stream=None):
    """qsa_split_touched_pages: page mark + masked split in one call."""
    arr, n = _sections(section_bytes)
    st = load_library().qsa_split_touched_pages(_ptr(indices), indices.numel(), _ptr(src_pool),
                                                _ptr(dst_pool), _ptr(mark), int(n_src_pages),
                                                int(src_page_size), int(dst_page_size), n, arr,
                                                _stream_ptr(stream))
    _check(st, "qsa_split_touched_pages")
    return dst_pool


def sparse_prefill_noalloc(q, k_cache, v_cache, indices, topk_len, scale: float, *, out=None,
                           lse=None, union_g: int = 0, stream=None):
    """Same as sparse_prefill, through qsa_sparse_prefill_noalloc: the library allocates
    nothing; union-mode scratch comes from its fixed NOALLOC_SCRATCH_BYTES device array.
    Calls needing more union scratch than that are refused (RuntimeError, QSA_ERR_WORKSPACE).
    Calls that overlap on the GPU share the array and race: keep them on one stream."""
    import torch
    lib = load_library()
    _require(q, torch.bfloat16, "q", 3)
    _require(k_cache, torch.bfloat16, "k_cache", 3)
    _require(v_cache, torch.bfloat16, "v_cache", 3)
    _require(indices, torch.int32, "indices", 2)
    _require(topk_len, torch.int32, "topk_len", 1)
    R, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((R, Hq), dtype=torch.float32, device=q.device)
    st = lib.qsa_sparse_prefill_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(indices),
                                        _ptr(topk_len), _ptr(out), _ptr(lse), R, Hq,
                                        k_cache.shape[1], D, indices.shape[1], float(scale),
                                        int(union_g), _stream_ptr(stream))
    if st == 3:
        raise RuntimeError(
            f"qsa_sparse_prefill_noalloc failed: QSA_ERR_WORKSPACE (union scratch of "
            f"{workspace_bytes(R, indices.shape[1], union_g)} bytes exceeds the fixed "
            f"{NOALLOC_SCRATCH_BYTES} bytes)")
    _check(st, "qsa_sparse_prefill_noalloc")
    return out, lse


def union_build(indices, topk_len, union_g: int, n_kv_slots: int = 0, want_sorted: bool = True,
                stream=None):
    """Runs qsa_union_build; returns (sorted [R, K] or None, union_idx, union_bits, union_len)."""
    import torch
    lib = load_library()
    _require(indices, torch.int32, "indices", 2)
    _require(topk_len, torch.int32, "topk_len", 1)
    R, K = indices.shape
    n_groups = -(-R // union_g)
    dev = indices.device
    srt = torch.empty((R, K), dtype=torch.int32, device=dev) if want_sorted else None
    uidx = torch.empty((n_groups, union_g * K), dtype=torch.int32, device=dev)
    ubits = torch.empty((n_groups, union_g * K), dtype=torch.uint8, device=dev)
    ulen = torch.empty((n_groups,), dtype=torch.int32, device=dev)
    st = lib.qsa_union_build(_ptr(indices), _ptr(topk_len), R, K, int(union_g), int(n_kv_slots),
                             _ptr(srt), _ptr(uidx), _ptr(ubits), _ptr(ulen), _stream_ptr(stream))
    _check(st, "qsa_union_build")
    return srt, uidx, ubits, ulen


GATHER_ENGINES = {"cpasync": 0, "tma": 1, "mixed": 2}


def probe_gather_ceiling(cache_rows, row_table, pieces_per_cta: int = 1500, engine: str = "tma",
                         stream=None) -> float:
    """Gather-ceiling probe (qsa_probe_gather_ceiling).  cache_rows: [n_rows, 256] bf16 view of a
    KV cache; row_table: [n_pieces, 128] int32 row numbers; engine: "tma" (tile::gather4) or
    "cpasync".  Returns GB/s over all SMs."""
    import torch
    lib = load_library()
    _require(cache_rows, torch.bfloat16, "cache_rows", 2)
    _require(row_table, torch.int32, "row_table", 2)
    ms = ctypes.c_float(0.0)
    st = lib.qsa_probe_gather_ceiling(_ptr(cache_rows), cache_rows.shape[0], _ptr(row_table),
                                      row_table.shape[0], int(pieces_per_cta),
                                      GATHER_ENGINES[engine], ctypes.byref(ms), _stream_ptr(stream))
    _check(st, "qsa_probe_gather_ceiling")
    sms = torch.cuda.get_device_properties(cache_rows.device).multi_processor_count
    return sms * pieces_per_cta * 32768 / (ms.value * 1e-3) / 1e9


def union_workspace_bytes(n_rows: int, topk: int, union_g: int) -> int:
    return int(load_library().qsa_union_workspace_bytes(n_rows, topk, union_g))


workspace_bytes = union_workspace_bytes


def select_geometry(n_qheads, n_kvheads, union_g, topk, head_dim, n_rows, num_sms=0) -> dict:
    g = Geometry()
    st = load_library().qsa_select_geometry(n_qheads, n_kvheads, union_g, topk, head_dim, n_rows,
                                            num_sms, ctypes.byref(g))
    _check(st, "qsa_select_geometry")
    return g.as_dict()


def select_geometry_status(n_qheads, n_kvheads, union_g, topk, head_dim, n_rows, num_sms) -> int:
    g = Geometry()
    return int(load_library().qsa_select_geometry(n_qheads, n_kvheads, union_g, topk, head_dim,
                                                  n_rows, num_sms, ctypes.byref(g)))


def counters() -> dict:
    c = Counters()
    load_library().qsa_get_counters(ctypes.byref(c))
    return c.as_dict()


def reset_counters():
    load_library().qsa_reset_counters()


def debug_stall_next_call():
    """Arm the failure-detection hook (qsa_debug_stall_next_call): the next attention call's
    bounded waits run out and it records a timeout in the device status word."""
    load_library().qsa_debug_stall_next_call()


def device_status(stream=None) -> int:
    v = ctypes.c_int32(0)
    st = load_library().qsa_get_device_status(_stream_ptr(stream), ctypes.byref(v))
    if st not in (0, 5):
        _check(st, "qsa_get_device_status")
    return int(v.value)


def version() -> str:
    return load_library().qsa_version().decode()
