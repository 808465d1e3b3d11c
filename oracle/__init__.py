"""CPU oracle for top-k sparse attention prefill -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct numpy (float64) restatements of what the sparse
prefill path computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference arm may import or run anything in this
package.  The product path (the CUDA library and its Python binding) never
imports it, and this package imports nothing from the product path: the two
share only the seeded input generators, which hold none of the method's
arithmetic and are passed in here as plain arrays.

Functions and the passages they follow:

* ``attention.sparse_prefill`` -- per-token sparse attention: for every query
  row, the query heads sharing one KV head attend over the gathered K/V rows
  of that row's selected slots (-1 = padding), scaled dot product, softmax,
  O and the per-head log-sum-exp.  Pages: "[QSA] Tune sm120 sparse prefill
  geometry" (Motivation: one program per query row, the [BLOCK_M, 256] fp32
  accumulator over up to 2051 gathered slots; Tests: the FP32 torch sparse
  attention reference, negative and out-of-range indices) and "DSA prefill
  ... triton_sparse_mla" (Motivation: online softmax in registers; Robustness:
  -1 marks an invalid slot, topk_length from metadata).
* ``union.sorted_rows`` / ``union.union_build`` -- the G-token union with its
  ownership bitmask ("DSA prefill ... triton_sparse_mla", Modifications: each
  row's selection is sorted by itself, a slot joins the list through the first
  row holding it and carries one bit per owning row; Accuracy Tests: the dedup
  contract -- every slot appears one time, its bits are the union of the rows
  that picked it, and padding is removed).
* ``union.union_attention`` -- attention of each token of a group over the
  union list restricted to its own ownership bit (same page: masking by the
  ownership bit leaves every token exactly its own slots, so union and
  per-token results agree).
* ``paged.sparse_prefill_paged`` -- the same attention when each row's slots
  are logical positions of its request, read through a page table with
  ragged request metadata ("DSA prefill ... triton_sparse_mla", Robustness:
  PAGED / RAGGED index transforms, valid length from the cache sequence
  lengths; "[QSA] Tune sm120 sparse prefill geometry": paged serving cache).
* ``mla.sparse_mla_prefill`` -- the MLA shape: one latent row per slot whose
  576 dims are the key and whose first 512 dims are the value, shared by every
  head ("DSA prefill ... triton_sparse_mla", Motivation and Speed Tests).
* ``pages.page_mark`` / ``pages.page_split`` -- the touched-page mark and the
  masked page split of "[SM120] Only split touched SWA pages in FlashMLA
  page-split kernel" (Modifications; the masked split equals the full split on
  every touched page and leaves the rest stale).
* ``fp8.sparse_prefill_fp8`` -- the same attention over an e4m3 KV cache with
  one scale per page and KV head, dequantised as e4m3(x) * scale ("DSA prefill
  ... triton_sparse_mla", Robustness and Accuracy Tests: dequantised rows).

Every function is pinned by ``tests/test_oracle_pins.py`` against facts that
do not come from this package: dense causal attention from a library routine
(sparse must equal dense when the selection is the whole causal prefix), a
library log-sum-exp, closed forms, invariances, and brute-force set
arithmetic for the union.
"""
from .attention import sparse_prefill, sparse_prefill_rows, valid_slots  # noqa: F401
from .union import sorted_rows, union_build, union_attention  # noqa: F401
from .paged import (sparse_prefill_paged, sparse_prefill_paged_rows,  # noqa: F401
                    physical_indices, request_of_rows)
from .mla import sparse_mla_prefill, sparse_mla_prefill_rows  # noqa: F401
from .pages import page_mark, page_split  # noqa: F401
from .fp8 import (e4m3_decode, dequantize, sparse_prefill_fp8,  # noqa: F401
                  sparse_prefill_fp8_rows)
