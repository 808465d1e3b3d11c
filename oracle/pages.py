"""Touched-page mark and page split, plain numpy -- TEST INFRASTRUCTURE ONLY (see the package
docstring).

Pages: "[SM120] Only split touched SWA pages in FlashMLA page-split kernel" (Modifications: a mark
pass sets mask[t // src_pbs] = 1 for every valid token index t, -1 skipped; the split copies a
page only when its mask is set, so the destination keeps stale data for the rest; the masked
result equals the full split on every touched page).

Page layout (the pages give none; plain reading): a page of P tokens holds its sections one
after another, section k being P x section_bytes[k] bytes, token-major.  Destination page
p * ratio + i holds source tokens i * dst_ps .. (i + 1) * dst_ps - 1 of page p.
"""
from __future__ import annotations

import numpy as np


def page_mark(indices, src_page_size: int, n_src_pages: int) -> np.ndarray:
    """uint8 [n_src_pages]: 1 where some valid index falls on the page."""
    mark = np.zeros(n_src_pages, dtype=np.uint8)
    for t in np.asarray(indices).reshape(-1):
        t = int(t)
        if t >= 0 and t // src_page_size < n_src_pages:
            mark[t // src_page_size] = 1
    return mark


def token_bytes_of(pool: np.ndarray, page: int, token: int, page_size: int, section_bytes):
    """Bytes of one token of one page, section by section (a list of byte arrays)."""
    page_bytes = page_size * sum(section_bytes)
    out, off = [], page * page_bytes
    for sb in section_bytes:
        out.append(pool[off + token * sb: off + (token + 1) * sb])
        off += page_size * sb
    return out


def page_split(src_pool: np.ndarray, dst_pool: np.ndarray, n_src_pages: int, src_page_size: int,
               dst_page_size: int, section_bytes, mark=None) -> np.ndarray:
    """A copy of dst_pool (uint8, flat) with every destination page of a marked source page
    (all pages when mark is None) written from src_pool, token by token."""
    ratio = src_page_size // dst_page_size
    dst = np.array(dst_pool, dtype=np.uint8, copy=True)
    dst_page_bytes = dst_page_size * sum(section_bytes)
    for p in range(n_src_pages):
        if mark is not None and not mark[p]:
            continue
        for i in range(ratio):
            q = p * ratio + i
            for u in range(dst_page_size):
                src_parts = token_bytes_of(src_pool, p, i * dst_page_size + u, src_page_size,
                                           section_bytes)
                off = q * dst_page_bytes
                for sb, part in zip(section_bytes, src_parts):
                    dst[off + u * sb: off + (u + 1) * sb] = part
                    off += dst_page_size * sb
    return dst
