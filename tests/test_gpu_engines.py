"""The two gather engines (TMA tile::gather4, the default, and cp.async 16-byte copies) against
each other and against the oracle, and the gather-ceiling probe for both (GPU only).

The engine is fixed per process (QSA_GATHER=cpasync selects cp.async), so the cp.async results are
computed in a child process and compared here: both engines put the same bytes in the same shared
memory tiles, so O and LSE must agree bit for bit."""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from helpers import to_device, assert_parity
from top_sparse_attention_row_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
from helpers import to_device
from top_sparse_attention_row_gb300 import binding as B, workloads as W
from engine_cases import cases
res = {{}}
for name, w, g in cases():
    q, k, v, idx, tl = to_device(w)
    out, lse = B.sparse_prefill(q, k, v, idx, tl, w.scale, union_g=g)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    res[name + "_out"] = out.view(torch.int16).cpu().numpy()
    res[name + "_lse"] = lse.cpu().numpy()
np.savez({path!r}, **res)
"""


@pytest.fixture(scope="module")
def B():
    from top_sparse_attention_row_gb300 import build, binding
    build.build()
    binding.load_library()
    return binding


def test_cpasync_engine_matches_tma_bitwise(B, tmp_path):
    import torch
    from engine_cases import cases
    path = str(tmp_path / "cpasync.npz")
    env = dict(os.environ, QSA_GATHER="cpasync")
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), path=path)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    other = np.load(path)
    for name, w, g in cases():
        q, k, v, idx, tl = to_device(w)
        out, lse = B.sparse_prefill(q, k, v, idx, tl, w.scale, union_g=g)
        torch.cuda.synchronize()
        assert B.device_status() == 0
        assert np.array_equal(out.view(torch.int16).cpu().numpy(), other[name + "_out"]), name
        assert np.array_equal(lse.cpu().numpy(), other[name + "_lse"], equal_nan=True), name
        O, L = oracle.sparse_prefill(w.q, w.k, w.v, w.indices, w.topk_len, w.scale)
        assert_parity(out, lse, O, L)


@pytest.mark.parametrize("engine", ["tma", "cpasync", "mixed"])
def test_gather_ceiling_probe(B, engine):
    import torch
    g = torch.Generator().manual_seed(7)
    n_rows = 1 << 16                                     # 32 MiB cache of 512-byte rows
    cache = torch.randn(n_rows, 256, generator=g).to(torch.bfloat16).cuda()
    table = torch.randint(0, n_rows, (512, 128), generator=g, dtype=torch.int32).cuda()
    gbs = B.probe_gather_ceiling(cache, table, pieces_per_cta=64, engine=engine)
    assert np.isfinite(gbs) and gbs > 100.0


def test_geometry_log_line(B):
    """QSA_LOG=1 prints the selected geometry, one line per attention call."""
    code = (f"import sys; sys.path.insert(0, {ROOT!r}); sys.path.insert(0, {os.path.join(ROOT, 'tests')!r})\n"
            "import torch\nfrom helpers import to_device\n"
            "from top_sparse_attention_row_gb300 import binding as B, workloads as W\n"
            "w = W.make_tiny(); q, k, v, idx, tl = to_device(w)\n"
            "B.sparse_prefill(q, k, v, idx, tl, w.scale); B.sparse_prefill(q, k, v, idx, tl, w.scale, union_g=2)\n"
            "torch.cuda.synchronize()\n")
    r = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, QSA_LOG="1"),
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stderr.splitlines() if l.startswith("qsa: d=256")]
    assert len(lines) == 2 and "union=1" in lines[0] and "union=2" in lines[1], r.stderr
