"""Reference append of new K/V rows into a paged cache -- TEST INFRASTRUCTURE.

Plain numpy, token by token, following the page-table slot rule: token t of
request i lives in page indices[indptr[i] + t / P] at slot t % P, K at index 0
and V at index 1 of the cache's second dimension ("FlashInfer, in depth",
section "The block-sparse page table"); appending a generated token writes
its K and V rows there (pyshine FlashInfer tour, "The Paged KV Cache Layer").
In the HND layout ([pages, 2, Hkv, P, D], "FlashInfer 完全拆解", section
接口层最容易踩的四个坑) the token's row of head h goes to [page, 0 or 1, h,
slot].  A token whose request, position or page falls outside the table is
skipped and reported.  Only tests and the benchmark's CPU leg use this module.
"""
from __future__ import annotations

import numpy as np


def append_kv(kv, k_new, v_new, batch_indices, positions, indptr, indices, last, page_size,
              layout="NHD"):
    """Return (new cache, list of skipped token numbers).

    kv: integer array (bf16 bit patterns or e4m3 bytes) [pages, 2, P, Hkv, D]
    (NHD) or [pages, 2, Hkv, P, D] (HND), not modified; k_new, v_new: the
    same dtype, [n, Hkv, D]; other arguments int sequences."""
    if layout not in ("NHD", "HND"):
        raise ValueError("layout must be 'NHD' or 'HND'")
    out = np.array(kv, copy=True)
    P = int(page_size)
    indptr = [int(x) for x in indptr]
    last = [int(x) for x in last]
    skipped = []
    for i in range(len(batch_indices)):
        b, pos = int(batch_indices[i]), int(positions[i])
        if not 0 <= b < len(last):
            skipped.append(i)
            continue
        n_pages = indptr[b + 1] - indptr[b]
        if n_pages < 1 or not 1 <= last[b] <= P:
            skipped.append(i)
            continue
        length = P * (n_pages - 1) + last[b]
        if not 0 <= pos < length:
            skipped.append(i)
            continue
        page = int(indices[indptr[b] + pos // P])
        if not 0 <= page < out.shape[0]:
            skipped.append(i)
            continue
        if layout == "NHD":
            out[page, 0, pos % P] = k_new[i]
            out[page, 1, pos % P] = v_new[i]
        else:
            for h in range(out.shape[2]):
                out[page, 0, h, pos % P] = k_new[i][h]
                out[page, 1, h, pos % P] = v_new[i][h]
    return out, skipped
