"""The C-ABI library builds, loads on a CPU-only machine and exports every declared symbol;
host-side validation and geometry selection (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from top_sparse_attention_row_gb300 import build, binding
    build.build()
    return binding.load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "qsa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qsa_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    from top_sparse_attention_row_gb300 import binding
    names = declared_functions()
    assert set(names) == set(binding.EXPORTED), names
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_status_strings(lib):
    from top_sparse_attention_row_gb300 import binding
    assert "sm_103a" in binding.version()
    for s in range(6):
        assert lib.qsa_status_string(s)


def test_selector_configs(lib):
    from top_sparse_attention_row_gb300 import binding as B
    g = B.select_geometry(6, 1, 0, 2051, 256, 8192, 152)
    assert g["n_pad"] == 16 and g["cols"] == 6 and g["union_g"] == 1 and g["grid"] == 152
    assert g["stages"] >= 4 and g["smem_bytes"] <= 232448 and g["n_items"] == 8192
    g = B.select_geometry(24, 2, 0, 2051, 256, 8192, 152)
    assert g["n_pad"] == 16 and g["cols"] == 12 and g["n_items"] == 16384
    g = B.select_geometry(8, 1, 4, 2048, 256, 8192, 152)
    assert g["union_g"] == 4 and g["n_pad"] == 32 and g["n_items"] == 2048
    g = B.select_geometry(8, 1, 2, 2048, 256, 8192, 152)
    assert g["union_g"] == 2 and g["n_pad"] == 16
    g = B.select_geometry(6, 1, 0, 128, 256, 256, 152)
    assert g["grid"] == 152 and g["n_items"] == 256
    g = B.select_geometry(6, 1, 0, 128, 256, 10, 152)
    assert g["grid"] == 10
    assert g["tmem_cols"] in (32, 64, 128, 256, 512) and g["tmem_cols"] >= 4 * g["n_pad"]


def test_selector_splits_small_calls(lib):
    """Per-token calls with fewer items than SMs share each item over a cluster of 2, 4 or 8
    CTAs (at most one tile each, tiles of <= 32 columns); everything else keeps split 1."""
    from top_sparse_attention_row_gb300 import binding as B
    expect = {1: 8, 7: 8, 19: 8, 20: 4, 32: 4, 38: 4, 39: 2, 64: 2, 76: 2, 77: 1, 128: 1, 8192: 1}
    for rows, split in expect.items():
        g = B.select_geometry(6, 1, 0, 2051, 256, rows, 152)
        assert g["split"] == split, (rows, g)
        assert g["grid"] == min(rows, 152 // split) * split and g["grid"] <= 152
        assert g["smem_bytes"] <= 232448 and (split == 1 or g["stages"] == 4)
    assert B.select_geometry(24, 2, 0, 2051, 256, 7, 152)["split"] == 8      # 14 items
    assert B.select_geometry(6, 1, 0, 300, 256, 7, 152)["split"] == 2       # 3 tiles a row
    assert B.select_geometry(6, 1, 0, 128, 256, 7, 152)["split"] == 1       # one tile
    assert B.select_geometry(6, 1, 4, 2051, 256, 7, 152)["split"] == 1      # union
    assert B.select_geometry(48, 1, 0, 2051, 256, 7, 152)["split"] == 1     # 48 columns


def test_selector_union_fallback_and_head_chunks(lib):
    from top_sparse_attention_row_gb300 import binding as B
    # 32 heads per KV group x G=4 = 128 columns > 64: falls back to per-token
    g = B.select_geometry(32, 1, 4, 2048, 256, 100, 152)
    assert g["union_g"] == 1 and g["n_pad"] == 32
    # 96 heads per group: two chunks of 48 columns
    g = B.select_geometry(96, 1, 0, 2048, 256, 100, 152)
    assert g["head_chunks"] == 2 and g["cols"] == 48 and g["n_pad"] == 48 and g["n_items"] == 200
    # 8 rows x 8 heads = 64 columns: the largest union tile; it keeps at least 4 stages
    g = B.select_geometry(8, 1, 8, 2048, 256, 100, 152)
    assert g["union_g"] == 8 and g["n_pad"] == 64 and g["stages"] >= 4
    assert g["smem_bytes"] <= 232448
    # odd union sizes are legal shapes in this kernel
    g = B.select_geometry(6, 1, 3, 2048, 256, 100, 152)
    assert g["union_g"] == 3 and g["n_pad"] == 32 and g["n_items"] == 34


@pytest.mark.parametrize("args,status", [
    ((6, 1, 0, 2051, 128, 10, 152), 2),     # head_dim != 256
    ((6, 4, 0, 2051, 256, 10, 152), 1),     # Hq % Hkv != 0
    ((6, 1, 9, 2051, 256, 10, 152), 1),     # union_g > 8
    ((6, 1, 0, 0, 256, 10, 152), 1),        # topk <= 0
    ((6, 1, 0, 2051, 256, -1, 152), 1),     # n_rows < 0
    ((6, 1, 0, 1 << 20, 256, 10, 152), 2),  # per-token slot list cannot fit shared memory
])
def test_selector_rejections(lib, args, status):
    from top_sparse_attention_row_gb300 import binding as B
    assert B.select_geometry_status(*args) == status


def test_entry_validation_before_any_cuda_call(lib):
    """Argument errors come back as statuses without touching the (absent) GPU."""
    f = lib.qsa_sparse_prefill
    fake = 1 << 20                     # 16-byte aligned non-null stand-in, never dereferenced
    assert f(None, fake, fake, fake, None, fake, None, 10, 6, 1, 256, 2051, 0.0625, 0, None) == 1
    assert f(fake + 2, fake, fake, fake, None, fake, None, 10, 6, 1, 256, 2051, 0.0625, 0, None) == 1
    assert f(fake, fake, fake, fake, None, fake, None, 10, 6, 1, 128, 2051, 0.0625, 0, None) == 2
    assert f(fake, fake, fake, fake, None, fake, None, 10, 6, 4, 256, 2051, 0.0625, 0, None) == 1
    assert f(fake, fake, fake, fake, None, fake, None, 10, 6, 1, 256, 2051, float("nan"), 0, None) == 1
    assert f(fake, fake, fake, fake, None, fake, None, 0, 6, 1, 256, 2051, 0.0625, 0, None) == 0
    ub = lib.qsa_union_build
    assert ub(None, None, 10, 16, 2, 0, None, fake, fake, fake, None) == 1
    assert ub(fake, None, 10, 16, 0, 0, None, fake, fake, fake, None) == 1
    assert ub(fake, None, 10, 1 << 16, 8, 0, None, fake, fake, fake, None) == 2
    pg = lib.qsa_sparse_prefill_paged
    #        q     k     v     idx   tl    cu    kvl   table out   lse   R   nreq ppr ps npages hq hkv d  topk scale  G
    assert pg(fake, fake, fake, fake, None, None, None, fake, fake, None, 10, 2, 4, 64, 0, 6, 1, 256, 64, 0.0625, 0, None) == 1
    assert pg(fake, fake, fake, fake, None, fake, None, None, fake, None, 10, 2, 4, 64, 0, 6, 1, 256, 64, 0.0625, 0, None) == 1
    assert pg(fake, fake, fake, fake, None, fake, None, fake, fake, None, 10, 0, 4, 64, 0, 6, 1, 256, 64, 0.0625, 0, None) == 1
    assert pg(fake, fake, fake, fake, None, fake, None, fake, fake, None, 10, 2, 0, 64, 0, 6, 1, 256, 64, 0.0625, 0, None) == 1
    assert pg(fake, fake, fake, fake, None, fake, None, fake, fake, None, 10, 2, 4, 0, 0, 6, 1, 256, 64, 0.0625, 0, None) == 1
    assert pg(fake, fake, fake, fake, None, fake, None, fake, fake, None, 10, 2, 4, 64, -1, 6, 1, 256, 64, 0.0625, 0, None) == 1
    assert pg(fake, fake, fake, fake, None, fake, None, fake, fake, None, 10, 2, 4, 64, 1 << 26, 6, 1, 256, 64, 0.0625, 0, None) == 2
    assert pg(fake, fake, fake, fake, None, fake, None, fake, fake, None, 10, 2, 4, 64, 0, 6, 1, 128, 64, 0.0625, 0, None) == 2
    assert pg(fake, fake, fake, fake, None, fake, None, fake, fake, None, 0, 2, 4, 64, 0, 6, 1, 256, 64, 0.0625, 0, None) == 0
    pr = lib.qsa_probe_gather_ceiling
    ms = ctypes.c_float(0.0)
    assert pr(fake, 1000, fake, 4, 10, 3, ctypes.byref(ms), None) == 1      # unknown engine
    assert pr(fake + 8, 1000, fake, 4, 10, 1, ctypes.byref(ms), None) == 1  # misaligned cache
    assert pr(fake, 1000, fake, 0, 10, 0, ctypes.byref(ms), None) == 1      # empty row table


def test_workspace_bytes(lib):
    from top_sparse_attention_row_gb300 import binding as B
    for args in ((8192, 2048, 4), (1023, 16, 3), (5, 7, 8), (100, 2048, 1), (0, 16, 4)):
        assert lib.qsa_union_workspace_bytes(*args) == lib.qsa_workspace_bytes(*args)
    assert B.workspace_bytes(8192, 2048, 1) == 0
    n = B.workspace_bytes(8192, 2048, 4)
    groups = 2048
    assert n >= groups * 4 * 2048 * 5 + groups * 4 and n % 256 == 0
    assert B.workspace_bytes(1023, 16, 4) >= 256 * 64 * 5


def test_counters_reset(lib):
    from top_sparse_attention_row_gb300 import binding as B
    B.reset_counters()
    assert all(v == 0 for v in B.counters().values())


def test_mla_selector(lib):
    """MLA geometry: N = heads (or G x heads) padded to 16/32, a 5-stage latent ring when it fits,
    union fallback past 32 columns, head chunks past 32 heads, d_qk/d_v other than 576/512
    unsupported."""
    from top_sparse_attention_row_gb300 import binding as B
    g = B.select_mla_geometry(8, 0, 2048, 8192, num_sms=152)
    assert (g["n_pad"], g["cols"], g["stages"], g["union_g"], g["tmem_cols"]) == (16, 8, 5, 1, 128)
    assert g["grid"] == 152 and g["n_items"] == 8192 and g["smem_bytes"] <= 232448
    g = B.select_mla_geometry(8, 4, 2048, 8192, num_sms=152)
    assert (g["n_pad"], g["cols"], g["union_g"], g["n_items"], g["tmem_cols"]) == (32, 32, 4, 2048, 256)
    assert g["stages"] == 4
    g = B.select_mla_geometry(16, 4, 2048, 100, num_sms=152)     # 64 columns: per-token instead
    assert g["union_g"] == 1 and g["n_pad"] == 16
    g = B.select_mla_geometry(40, 0, 2048, 10, num_sms=152)      # two chunks of 20 heads
    assert g["head_chunks"] == 2 and g["cols"] == 20 and g["n_pad"] == 32 and g["n_items"] == 20
    sel = lib.qsa_select_mla_geometry
    out = B.Geometry()
    assert sel(8, 0, 2048, 512, 512, 10, 152, ctypes.byref(out)) == 2
    assert sel(8, 0, 2048, 576, 256, 10, 152, ctypes.byref(out)) == 2
    assert sel(0, 0, 2048, 576, 512, 10, 152, ctypes.byref(out)) == 1
    assert sel(8, 0, 1 << 16, 576, 512, 10, 152, ctypes.byref(out)) == 2   # slot list too large
    f = lib.qsa_sparse_mla_prefill
    fake = 1 << 20
    assert f(None, fake, fake, None, fake, None, 10, 8, 576, 512, 2048, 0.04, 0, 0, None) == 1
    assert f(fake, fake + 8, fake, None, fake, None, 10, 8, 576, 512, 2048, 0.04, 0, 0, None) == 1
    assert f(fake, fake, fake, None, fake, None, 10, 8, 576, 256, 2048, 0.04, 0, 0, None) == 2
    assert f(fake, fake, fake, None, fake, None, 0, 8, 576, 512, 2048, 0.04, 0, 0, None) == 0


def test_page_split_validation(lib):
    """Page mark / split argument errors come back before any GPU work."""
    fake = 1 << 20
    secs = (ctypes.c_int32 * 3)(512, 16, 128)
    bad = (ctypes.c_int32 * 2)(512, 8)                     # not a multiple of 16
    sp = lib.qsa_page_split
    assert sp(None, fake, None, 10, 256, 64, 3, secs, None) == 1
    assert sp(fake, fake, None, 10, 256, 96, 3, secs, None) == 1          # 256 % 96 != 0
    assert sp(fake, fake, None, 10, 256, 64, 2, bad, None) == 1
    assert sp(fake, fake, None, 10, 256, 64, 0, secs, None) == 1
    assert sp(fake, fake, None, 10, 256, 64, 9, secs, None) == 1
    assert sp(fake + 4, fake, None, 10, 256, 64, 3, secs, None) == 1
    assert sp(fake, fake, None, 1 << 30, 256, 64, 3, secs, None) == 2     # grid past 2^31
    assert sp(fake, fake, None, 0, 256, 64, 3, secs, None) == 0
    pm = lib.qsa_page_mark
    assert pm(fake, 10, 256, 10, None, None) == 1
    assert pm(None, 10, 256, 10, fake, None) == 1
    assert pm(fake, 10, 0, 10, fake, None) == 1
    assert pm(fake, 10, 256, 0, fake, None) == 0
    st = lib.qsa_split_touched_pages
    assert st(fake, 10, fake, fake, None, 10, 256, 64, 3, secs, None) == 1
    assert st(fake, 10, fake, fake, fake, 10, 256, 48, 3, secs, None) == 1


def test_fp8_entry_validation(lib):
    f = lib.qsa_sparse_prefill_fp8
    fake = 1 << 20
    #        q     k     v     ks    vs    ps  idx   tl    out   lse   R   hq hkv d    topk scale  G  nkv
    assert f(fake, fake, fake, None, fake, 64, fake, None, fake, None, 10, 6, 1, 256, 2051, 0.0625, 0, 0, None) == 1
    assert f(fake, fake, fake, fake, None, 64, fake, None, fake, None, 10, 6, 1, 256, 2051, 0.0625, 0, 0, None) == 1
    assert f(fake, fake, fake, fake, fake, 0, fake, None, fake, None, 10, 6, 1, 256, 2051, 0.0625, 0, 0, None) == 1
    assert f(fake, fake + 8, fake, fake, fake, 64, fake, None, fake, None, 10, 6, 1, 256, 2051, 0.0625, 0, 0, None) == 1
    assert f(fake, fake, fake, fake, fake, 64, fake, None, fake, None, 10, 6, 1, 128, 2051, 0.0625, 0, 0, None) == 2
    assert f(fake, fake, fake, fake, fake, 64, fake, None, fake, None, 0, 6, 1, 256, 2051, 0.0625, 0, 0, None) == 0


def _params(name):
    src = open(os.path.join(ROOT, "include", "qsa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    m = re.search(r"\b" + name + r"\s*\(([^)]*)\)\s*;", src)
    assert m, name
    return [re.split(r"[\s*]+", p.strip())[-1] for p in m.group(1).split(",") if p.strip()]


def test_boundary_entry_points_and_argument_lists(lib):
    """Every call of the boundary is exported under its name, and the attention entry keeps the
    argument list of the operation: q, caches, indices, topk_len, outputs, sizes, scale, union size
    and stream, in that order; the extended entry adds the slot count, the caller workspace and a
    forced geometry before the stream."""
    for name in ("qsa_sparse_prefill", "qsa_sparse_prefill_ex", "qsa_union_workspace_bytes",
                 "qsa_union_build", "qsa_select_geometry", "qsa_get_counters", "qsa_reset_counters",
                 "qsa_status_string", "qsa_version", "qsa_get_device_status"):
        assert hasattr(lib, name), name
    main = ["q", "k_cache", "v_cache", "indices", "topk_len", "out", "lse", "n_rows", "n_qheads",
            "n_kvheads", "head_dim", "topk", "scale", "union_g", "stream"]
    assert _params("qsa_sparse_prefill") == main
    assert _params("qsa_sparse_prefill_ex") == main[:-1] + ["n_kv_slots", "workspace",
                                                            "workspace_bytes", "forced", "stream"]
    assert _params("qsa_union_workspace_bytes") == ["n_rows", "topk", "union_g"]
    # the selector also takes the KV head count (work items are row groups x KV heads) and the SM
    # count (so host-only callers choose it; <= 0 asks the current device)
    assert _params("qsa_select_geometry") == ["n_qheads", "n_kvheads", "union_g", "topk",
                                              "head_dim", "n_rows", "num_sms", "out"]
