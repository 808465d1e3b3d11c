"""qsa_sparse_prefill_noalloc: the entry point for callers that must not allocate device
memory (GPU only).

Its union-mode scratch is a fixed array the library owns, so two calls in a row reuse the same
memory; each must match the allocating entry point within the parity bounds.  This file is
named to be collected last, so a run that stops at the first failure has already run every
other test; it also passes on its own in a fresh process."""
import os
import subprocess
import sys

import numpy as np
import pytest

from helpers import to_device, compare, O_ATOL, LSE_RTOL
from top_sparse_attention_row_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from top_sparse_attention_row_gb300 import build, binding
    build.build()
    binding.load_library()
    return binding


def _walk(n_rows, topk, seed):
    rng = np.random.default_rng(seed)
    q = W.randn_bf16(rng, (n_rows, 8, 256))
    k = W.randn_bf16(rng, (n_rows, 1, 256))
    v = W.randn_bf16(rng, (n_rows, 1, 256))
    idx = W.random_walk_indices(rng, n_rows, topk)
    return W.Workload("walk", q, k, v, idx, None, 1.0 / 16.0, np.arange(n_rows))


def _check_same(out_a, lse_a, out_b, lse_b):
    dO, dL, mism = compare(out_a, lse_a, out_b.float().cpu().numpy(), lse_b.cpu().numpy())
    assert mism == 0 and dO <= O_ATOL and dL <= LSE_RTOL, (dO, dL, mism)


@pytest.mark.parametrize("union_g", [2, 4, 0])
def test_noalloc_matches_allocating_entry_twice(B, union_g):
    import torch
    ws = [_walk(613, 384, seed=50 + union_g), _walk(401, 384, seed=60 + union_g)]
    for w in ws:                                       # two calls in a row on the shared array
        q, k, v, idx, tl = to_device(w)
        ref_out, ref_lse = B.sparse_prefill(q, k, v, idx, tl, w.scale, union_g=union_g)
        out, lse = B.sparse_prefill_noalloc(q, k, v, idx, tl, w.scale, union_g=union_g)
        torch.cuda.synchronize()
        assert B.device_status() == 0
        _check_same(out, lse, ref_out, ref_lse)


def test_noalloc_refuses_calls_beyond_its_scratch(B):
    import torch
    R, K = 8192, 2048                                  # union workspace ~84 MB > 32 MiB
    assert B.workspace_bytes(R, K, 2) > B.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((R, 8, 256), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((R, 1, 256), dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros((R, K), dtype=torch.int32, device="cuda")
    B.reset_counters()
    with pytest.raises(RuntimeError, match="WORKSPACE"):
        B.sparse_prefill_noalloc(q, kv, kv, idx, None, 0.0625, union_g=2)
    assert B.counters()["kernel_launches"] == 0       # refused before anything was enqueued


def test_noalloc_per_token_first_in_a_fresh_process(B):
    """A per-token call that comes first in a process needs no scratch: it runs without looking
    the array up, and a union call after it still matches the allocating entry."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = (
        "import sys, torch\n"
        f"sys.path[:0] = [{root!r}, {os.path.join(root, 'tests')!r}]\n"
        "from top_sparse_attention_row_gb300 import binding as B, workloads as W\n"
        "from helpers import to_device, compare\n"
        "B.load_library()\n"
        "w = W.make_tiny(); q, k, v, idx, tl = to_device(w)\n"
        "for G in (0, 2):\n"
        "    o, l = B.sparse_prefill_noalloc(q, k, v, idx, tl, w.scale, union_g=G)\n"
        "    ro, rl = B.sparse_prefill(q, k, v, idx, tl, w.scale, union_g=G)\n"
        "    torch.cuda.synchronize()\n"
        "    dO, dL, mism = compare(o, l, ro.float().cpu().numpy(), rl.cpu().numpy())\n"
        "    assert mism == 0 and dO <= 2e-2 and dL <= 1e-3, (G, dO, dL, mism)\n"
        "assert B.device_status() == 0\n"
        "print('ok')\n")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stderr[-2000:]
