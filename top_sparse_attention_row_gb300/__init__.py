"""Top-k sparse attention prefill for GB300 (sm_103a).

The compute path is the C-ABI library ``libqsa.so`` built from ``csrc/``;
``binding`` marshals torch tensors into it.  Import ``binding`` (or call
``load_library``) explicitly: importing this package alone loads nothing, so
the seeded workload generators stay usable on machines without the library.
"""
__all__ = ["binding", "workloads"]
