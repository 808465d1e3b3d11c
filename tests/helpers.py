"""Shared test plumbing: workload -> device tensors, oracle comparison with the stated bounds."""
import numpy as np

O_ATOL = 2e-2          # max-abs bound on O against the oracle ("[QSA] ..." Tests: atol 2e-2)
LSE_RTOL = 1e-3        # |dLSE| <= 1e-3 * max(1, |LSE|); -inf must match exactly


def to_device(w, device="cuda"):
    import torch
    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)
    q, k, v = bf(w.q), bf(w.k), bf(w.v)
    idx = torch.from_numpy(np.ascontiguousarray(w.indices, dtype=np.int32)).to(device)
    tl = None if w.topk_len is None else torch.from_numpy(np.ascontiguousarray(w.topk_len, dtype=np.int32)).to(device)
    return q, k, v, idx, tl


def compare(out, lse, O_ref, L_ref, rows=None):
    """Returns (max |dO|, max scaled |dLSE|, LSE -inf mismatches) for the given rows."""
    o = out.float().cpu().numpy()
    l = lse.float().cpu().numpy()
    if rows is not None:
        o, l = o[rows], l[rows]
    dO = float(np.max(np.abs(o - O_ref))) if o.size else 0.0
    inf_ref, inf_got = np.isneginf(L_ref), np.isneginf(l)
    mism = int(np.sum(inf_ref != inf_got))
    fin = ~inf_ref & ~inf_got
    dL = float(np.max(np.abs(l[fin] - L_ref[fin]) / np.maximum(1.0, np.abs(L_ref[fin])))) if fin.any() else 0.0
    return dO, dL, mism


def assert_parity(out, lse, O_ref, L_ref, rows=None, what=""):
    dO, dL, mism = compare(out, lse, O_ref, L_ref, rows)
    assert mism == 0, f"{what}: {mism} LSE -inf mismatches"
    assert dO <= O_ATOL, f"{what}: max |dO| = {dO:.3e} > {O_ATOL}"
    assert dL <= LSE_RTOL, f"{what}: max rel |dLSE| = {dL:.3e} > {LSE_RTOL}"
    return dO, dL
