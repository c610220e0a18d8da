"""Reference restatement of the decode planner -- TEST INFRASTRUCTURE ONLY.

A slow, plain-Python statement of the host scheduler's steps, written
independently of the C++ planner inside the CUDA library.  Tests compare the
library's schedule with this one integer for integer.  Only tests, the
package smoke check and the benchmark's CPU-baseline leg import it.

Steps and where they come from:

P0  table check and lengths: indptr starts at 0 and is strictly increasing
    (every request owns at least one page), 1 <= last_page_len <= P, page ids
    inside the pool; l_i = P (n_i - 1) + r_i
    ("FlashInfer 完全拆解", section 页表就是一张块稀疏矩阵;
     "FlashInfer, in depth", section "Failure modes in production").
P1  chunk size: with one query token per request and the GQA group folded
    into the work unit, the work bound is L_kv = ceil(sum_i l_kv(i) / N_CTA)
    ("FlashInfer 完全拆解", section 先切长 KV，再做最长任务优先分配).  The
    chunk is L_kv rounded up to whole pages (a page is the block column),
    and never below a floor, so short requests are not split ("FlashInfer,
    in depth", section "Load balancing with split-KV"; "FlashInfer 完全拆解",
    section Split-KV 解决的是并行度).  Reading taken where the pages leave it
    open: the candidates L_kv, L_kv/2 and L_kv/4 are each scheduled and the
    one with the smallest predicted makespan wins (ties: the larger chunk).
P1' chunk size by search (variant): the largest chunk that still fills the
    GPU (pyshine FlashInfer tour, "Planning on the Host, Executing on the
    Device", where the prefill planner binary-searches it).  Reading
    taken: "fills the GPU" = the split gives at least N_CTA work items; the
    chunk is a whole number of pages and never below the floor (the floor
    when even it gives fewer items).  Stated here as a scan down from the
    longest request; the library binary-searches the same predicate, which
    only falls as the chunk grows.
P2  split and cost: a request longer than the chunk becomes chunks
    [k c, min((k+1) c, l)); cost C = alpha * l_q + beta * l_kv with l_q = 1
    and beta = 1, so C = alpha + len (same section, the cost model).
P3  LPT: items in descending cost (ties: request, then chunk, ascending), each
    given to the CTA with the least accumulated cost (ties: lowest CTA id)
    (same section).
P4  reduction map: split requests get contiguous partial slots in chunk
    order; unsplit items write through to the output (slot -1)
    ("FlashInfer 完全拆解", sections 先切长 KV (fixed reduction map, no
    atomics) and Split-KV 解决的是并行度 (writethrough)).  Each item names its
    pages by the index of its first page in the CSR indices array, which is
    passed on unchanged ("FlashInfer, in depth", "The block-sparse page
    table": request i owns indices[indptr[i]:indptr[i+1]]).
"""
from __future__ import annotations

import heapq
from dataclasses import dataclass

import numpy as np


class TableError(ValueError):
    pass


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def _round_up(a: int, b: int) -> int:
    return _ceil_div(a, b) * b


def lengths(indptr, last, indices, page_size: int, num_pages: int):
    """P0: validate the CSR table and return per-request token counts."""
    indptr = [int(x) for x in indptr]
    last = [int(x) for x in last]
    batch = len(last)
    if len(indptr) != batch + 1:
        raise TableError("indptr must have batch + 1 entries")
    if batch and indptr[0] != 0:
        raise TableError("indptr[0] must be 0")
    lens = []
    for i in range(batch):
        n = indptr[i + 1] - indptr[i]
        if n < 1:
            raise TableError(f"request {i} owns no page")
        r = last[i]
        if not 1 <= r <= page_size:
            raise TableError(f"last_page_len[{i}] = {r} outside 1..{page_size}")
        lens.append(page_size * (n - 1) + r)
    if batch:
        idx = np.asarray(indices[: indptr[-1]], dtype=np.int64)
        if idx.shape[0] != indptr[-1]:
            raise TableError("indices shorter than indptr[-1]")
        if idx.size and (idx.min() < 0 or idx.max() >= num_pages):
            raise TableError("page id outside the pool")
    return lens


@dataclass
class Plan:
    chunk: int
    makespan: int
    cta_indptr: list          # [n_cta + 1]
    items: list               # per item, queue order: (first request, tok_begin, tok_end,
    #                           dst_slot, first page index, requests, slot stride)
    units: list               # per split request: (req, n_chunks)
    merge_indptr: list        # [n_units + 1]
    page_list: list           # the CSR page ids, as given
    lens: list                # per block (per request without grouping)
    heads: list = None        # per item: its KV head (per-head plans), else 0

    @property
    def n_items(self):
        return len(self.items)

    @property
    def n_slots(self):
        return self.merge_indptr[-1] if self.merge_indptr else 0


def _split(lens, chunk, alpha):
    """P2: (cost, req, chunk_index, tok_begin, tok_end) per item."""
    items = []
    for i, l in enumerate(lens):
        k = 0
        t = 0
        while t < l:
            e = min(t + chunk, l)
            items.append((alpha + (e - t), i, k, t, e))
            t = e
            k += 1
    return items


def _lpt(items, n_cta):
    """P3: longest-processing-time-first onto n_cta queues."""
    order = sorted(items, key=lambda it: (-it[0], it[1], it[2]))
    heap = [(0, c) for c in range(n_cta)]
    queues = [[] for _ in range(n_cta)]
    for it in order:
        load, c = heapq.heappop(heap)
        queues[c].append(it)
        heapq.heappush(heap, (load + it[0], c))
    loads = [0] * n_cta
    for load, c in heap:
        loads[c] = load
    return queues, max(loads) if loads else 0


def n_split_items(lens, chunk):
    """Number of work items the split at ``chunk`` tokens gives."""
    return sum(_ceil_div(l, chunk) for l in lens)


def search_chunk(lens, *, page_size: int, n_cta: int, floor: int) -> int:
    """P1': the largest multiple of the page size, not below ``floor`` (a page
    multiple), whose split gives at least n_cta items; ``floor`` when none
    does."""
    top = max(_round_up(max(lens), page_size), floor) if lens else floor
    c = top
    while c > floor:
        if n_split_items(lens, c) >= n_cta:
            return c
        c -= page_size
    return floor


def plan(indptr, indices, last, *, page_size: int, num_pages: int, n_cta: int,
         alpha: int, min_chunk_tokens: int, chunk_divisors=(1, 2, 4), group_indptr=None,
         rows: int = 1, chunk_rule: str = "closed", per_head: int = 1) -> Plan:
    """Schedule a decode step.  Without ``group_indptr`` the table has one row
    per request.  With it (a shared-prefix level, "FlashInfer 完全拆解",
    section Composable Format) the table has one row per group, requests
    group_indptr[j] .. group_indptr[j+1]-1 share group j's pages, and each
    group's requests are cut into blocks of ``rows`` consecutive requests; a
    work item covers one block.  With ``per_head`` = Hkv (the dense-prefix
    kernel, whose tile is one KV head's rows of a block) the unit of work is
    (block, KV head), units ordered block-major, and an item covers one
    head of one block."""
    row_lens = lengths(indptr, last, indices, page_size, num_pages)
    P = page_size
    if group_indptr is None:
        blocks = [(i, 1, i) for i in range(len(row_lens))]     # (first request, n, table row)
    else:
        gi = [int(x) for x in group_indptr]
        if len(gi) != len(row_lens) + 1 or (gi and gi[0] != 0):
            raise TableError("group_indptr must have one entry per group + 1, starting at 0")
        blocks = []
        for j in range(len(row_lens)):
            if gi[j + 1] <= gi[j]:
                raise TableError(f"group {j} has no request")
            for r in range(gi[j], gi[j + 1], rows):
                blocks.append((r, min(rows, gi[j + 1] - r), j))
    lens = [row_lens[b[2]] for b in blocks]
    # units of work: (block, head), block-major
    ulens = [l for l in lens for _ in range(per_head)]
    W = sum(ulens)
    L = _ceil_div(W, n_cta)
    floor = _round_up(max(min_chunk_tokens, 1), P)
    cands = []
    if chunk_rule == "search":
        cands.append(search_chunk(ulens, page_size=P, n_cta=n_cta, floor=floor))
    elif chunk_rule == "closed":
        for k in chunk_divisors:
            c = max(_round_up(_ceil_div(L, k), P), floor)
            if c not in cands:
                cands.append(c)
    else:
        raise ValueError("chunk_rule must be 'closed' or 'search'")
    best = None
    for c in cands:
        queues, makespan = _lpt(_split(ulens, c, alpha), n_cta)
        if best is None or makespan < best[1]:
            best = (c, makespan, queues)
    chunk, makespan, queues = best

    # P4: reduction map: each request of a split block is a unit with one
    # partial slot per chunk; units in ascending request order
    n_chunks = [_ceil_div(l, chunk) for l in lens]
    units = []
    merge_indptr = [0]
    block_slot = {}
    for bi, (r0, n, row) in enumerate(blocks):
        if n_chunks[bi] > 1:
            block_slot[bi] = merge_indptr[-1]
            for r in range(r0, r0 + n):
                units.append((r, n_chunks[bi]))
                merge_indptr.append(merge_indptr[-1] + n_chunks[bi])

    cta_indptr = [0]
    items = []
    heads = []
    indptr = [int(x) for x in indptr]
    for q in queues:
        for cost, u, k, tb, te in q:
            bi, head = divmod(u, per_head)
            heads.append(head)
            r0, n, row = blocks[bi]
            split = bi in block_slot
            dst = block_slot[bi] + k if split else -1
            # page reference: index (into the CSR indices) of the item's first
            # page; request r0 + i of the block writes slot dst + i * stride
            items.append((r0, tb, te, dst, indptr[row] + tb // P, n,
                          n_chunks[bi] if split else 0))
        cta_indptr.append(len(items))
    page_list = [int(x) for x in indices[: indptr[-1] if indptr else 0]]
    return Plan(chunk, makespan, cta_indptr, items, units, merge_indptr,
                page_list, lens, heads)
