"""Sparse attention prefill over an FP8 (e4m3) KV cache with per-page scales, float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Pages: "DSA prefill ... triton_sparse_mla" (Robustness: the Triton kernel refuses a packed FP8
pool; Accuracy Tests: flashinfer reads the FP8 cache together with its scales, while the
Triton kernel is handed rows already dequantised to bf16).  The plain reading of "dequantised": the value of cache byte x
at slot s, KV head h is e4m3(x) * scale[s // page_size, h], and attention is the plain
definition (attention.sparse_prefill) on those values.

e4m3 (the 8-bit float with 1 sign, 4 exponent bits of bias 7, 3 mantissa bits, no infinities):
    exponent 0          -> (-1)^s * m/8 * 2^-6          (zero and subnormals)
    exponent 15, m = 7  -> NaN
    otherwise           -> (-1)^s * (1 + m/8) * 2^(e-7)  (largest finite 448)
"""
from __future__ import annotations

import numpy as np

from .attention import sparse_prefill_rows


def e4m3_decode(codes) -> np.ndarray:
    """uint8 codes -> float64 values, from the bit layout above."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def dequantize(cache, scale, page_size: int) -> np.ndarray:
    """cache [S, Hkv, D] e4m3 codes, scale [pages, Hkv] -> float64 [S, Hkv, D]."""
    vals = e4m3_decode(cache)
    S = vals.shape[0]
    page = np.arange(S) // page_size
    return vals * np.asarray(scale, dtype=np.float64)[page][:, :, None]


def sparse_prefill_fp8_rows(q, k8, v8, k_scale, v_scale, page_size: int, indices, topk_len,
                            scale: float, rows, n_kv_slots: int = 0):
    k = dequantize(k8, k_scale, page_size)
    v = dequantize(v8, v_scale, page_size)
    return sparse_prefill_rows(q, k, v, indices, topk_len, scale, rows, n_kv_slots)


def sparse_prefill_fp8(q, k8, v8, k_scale, v_scale, page_size: int, indices, topk_len,
                       scale: float, n_kv_slots: int = 0):
    return sparse_prefill_fp8_rows(q, k8, v8, k_scale, v_scale, page_size, indices, topk_len,
                                   scale, np.arange(q.shape[0]), n_kv_slots)
