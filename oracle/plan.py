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
    # partial slot per chunk, in chunk order; units longest first (most
    # chunks, ties by request), the pages' longest-first rule applied to the
    # merge's tasks
    n_chunks = [_ceil_div(l, chunk) for l in lens]
    units = []
    merge_indptr = [0]
    block_slot = {}
    split_blocks = sorted((bi for bi in range(len(blocks)) if n_chunks[bi] > 1),
                          key=lambda bi: (-n_chunks[bi], bi))
    for bi in split_blocks:
        r0, n, row = blocks[bi]
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


@dataclass
class CascadePlan:
    n_pre: int                # CTAs [0, n_pre) run the prefix items
    chunk_pre: int
    chunk_suf: int
    makespan: int             # in suffix-token units (the larger level's)
    cta_indptr: list
    items: list               # (first request, tok_begin, tok_end, dst, first page index,
    #                           requests, slot stride, KV head), queue order
    units: list               # (request, slots) for every request
    merge_indptr: list
    page_list: list           # prefix table's page ids, then the suffix table's


def _level(ulens, n, page_size, floor, alpha):
    """One level of a cascade plan: closed-form chunk candidates (the work
    bound over the level's n CTAs, and its half), page-rounded and not below
    the floor; the smaller LPT makespan wins (ties: the larger chunk)."""
    bound = _ceil_div(sum(ulens), n)
    best = None
    prev = None
    for k in (1, 2):
        c = max(_round_up(_ceil_div(bound, k), page_size), floor)
        if c == prev:
            continue
        prev = c
        if best is not None:
            # a makespan is at least the costliest item and the mean load:
            # a candidate that cannot beat the best strictly is not scheduled
            n_it = sum(_ceil_div(l, c) for l in ulens)
            lb = max(alpha + max(min(l, c) for l in ulens),
                     _ceil_div(sum(ulens) + alpha * n_it, n))
            if lb >= best[1]:
                continue
        queues, span = _lpt(_split(ulens, c, alpha), n)
        if best is None or span < best[1]:
            best = (c, span, queues)
    return best


def _prefix_level(block_lens, hkv, n, page_size, floor, alpha):
    """The prefix level of a cascade plan on a budget of n CTAs: at most one
    item per CTA.  Every block starts with one chunk per KV head; while hkv
    more CTAs are left, the block with the longest chunk (ties: the first)
    gets one more chunk per head, unless its chunk would fall below the
    floor; then each block keeps the fewest chunks that stay within the
    longest chunk (more would not shorten the level).  Chunks are
    page-rounded; item j goes to CTA j.  With more heads than CTAs the
    (block, head) units stay whole and LPT places them.
    Returns (span, queues, chunk per block, CTAs used)."""
    nb = len(block_lens)
    if nb * hkv > n:
        top = max(max(block_lens), 1)
        units = [l for l in block_lens for _ in range(hkv)]
        queues, span = _lpt(_split(units, top, alpha), n)
        return span, queues, [top] * nb, n
    m = [1] * nb
    chunk = [_round_up(l, page_size) for l in block_lens]
    budget = n - nb * hkv
    while budget >= hkv:
        b = max(range(nb), key=lambda i: (chunk[i], -i))
        nxt = _round_up(_ceil_div(block_lens[b], m[b] + 1), page_size)
        if nxt < floor:
            break
        m[b] += 1
        chunk[b] = nxt
        budget -= hkv
    # chunks that do not lower the level's longest one are given back: every
    # block keeps the fewest chunks whose length stays within it
    top = max(chunk)
    for b in range(nb):
        while m[b] > 1 and _round_up(_ceil_div(block_lens[b], m[b] - 1), page_size) <= top:
            m[b] -= 1
        chunk[b] = _round_up(_ceil_div(block_lens[b], m[b]), page_size)
    queues, span = [], 0
    for b, l in enumerate(block_lens):
        for h in range(hkv):
            k, t = 0, 0
            while t < l:
                e = min(t + chunk[b], l)
                queues.append([(alpha + e - t, b * hkv + h, k, t, e)])
                span = max(span, alpha + e - t)
                t, k = e, k + 1
    return span, queues, chunk, len(queues)


def plan_cascade(group_indptr, prefix, suffix, *, page_size: int, num_pages: int, n_cta: int,
                 hkv: int, rows: int, alpha: int, prefix_alpha: int, prefix_cost16: int,
                 suffix_floor: int, prefix_floor: int = 128) -> CascadePlan:
    """A decode step whose requests share prefix pages in groups and each own
    a suffix ("FlashInfer, in depth", "Prefill, masks and shared prefixes" and
    "Cascades, Merges, and the Autotuner": the shared part once for all
    queries, each suffix apart, one merge of the two states; "FlashInfer
    完全拆解", Composable Format), planned as one schedule:

    * prefix work units are (block of up to ``rows`` requests of a group,
      KV head), block-major; suffix units are the requests;
    * the grid is cut at n_pre: CTAs [0, n_pre) take the prefix level (at
      most one item each, see _prefix_level), the rest the suffix level,
      split at its own closed-form chunk and scheduled by LPT (P1-P3 above)
      on its own CTAs;
    * prefix items cost (prefix_alpha + tokens) * prefix_cost16 / 16 in
      suffix-token units, suffix items alpha + tokens; the prefix budget
      starts where each level gets CTAs in proportion to its total cost (in
      steps of hkv above one CTA per unit when the grid allows, rounded to
      the nearest step); budgets are compared by the predicted makespan,
      ties by the sum of the two levels' makespans; the search moves from
      the start toward its better neighbour (the next budget either way
      whose prefix level differs), if that one is strictly better, and on
      from neighbour to neighbour while the budget keeps improving
      strictly; the suffix gets every CTA the prefix items do not use;
    * every request is a unit of the reduction map whose slots are its
      prefix chunks then its suffix chunks (all items write partial states).
    """
    P = page_size
    gi = [int(x) for x in group_indptr]
    p_ip, p_ix, p_last = prefix
    s_ip, s_ix, s_last = suffix
    pre_len = lengths(p_ip, p_last, p_ix, P, num_pages)
    suf_len = lengths(s_ip, s_last, s_ix, P, num_pages)
    if len(gi) != len(pre_len) + 1 or (gi and gi[0] != 0):
        raise TableError("group_indptr must have one entry per group + 1, starting at 0")
    batch = gi[-1] if gi else 0
    if len(suf_len) != batch:
        raise TableError("one suffix row per request")
    blocks = []                          # (first request, n, group)
    for j in range(len(pre_len)):
        if gi[j + 1] <= gi[j]:
            raise TableError(f"group {j} has no request")
        for r in range(gi[j], gi[j + 1], rows):
            blocks.append((r, min(rows, gi[j + 1] - r), j))
    block_of = {}
    for b, (r0, n, j) in enumerate(blocks):
        for r in range(r0, r0 + n):
            block_of[r] = b
    block_lens = [pre_len[j] for (_, _, j) in blocks]
    pre_cost = sum(hkv * (prefix_alpha + l) * prefix_cost16 for l in block_lens)
    suf_cost = sum((alpha + l) * 16 for l in suf_len)
    floor_s = _round_up(max(suffix_floor, 1), P)
    floor_p = _round_up(prefix_floor, P)
    best = None
    if batch:
        units = len(blocks) * hkv
        split = units <= n_cta - 1
        base, step = (units, hkv) if split else (1, 1)
        j_max = (n_cta - 1 - base) // step
        prop = (n_cta * pre_cost + (pre_cost + suf_cost) // 2) // (pre_cost + suf_cost)
        j0 = min(max((max(prop - base, 0) + step // 2) // step, 0), j_max)

        def schedule(j):
            pre = _prefix_level(block_lens, hkv, base + step * j, P, floor_p, prefix_alpha)
            suf = _level(suf_len, n_cta - pre[3], P, floor_s, alpha)
            p_span, s_span = pre[0] * prefix_cost16, suf[1] * 16
            return ((max(p_span, s_span), p_span + s_span), j, pre, suf)

        def used(j):                      # CTAs the prefix level takes at budget j
            return _prefix_level(block_lens, hkv, base + step * j, P, floor_p, prefix_alpha)[3]

        def neighbour(j, d):
            """The next budget from j in direction d whose prefix level
            differs (budgets between give the same plan), or None."""
            c = used(j)
            k = j + d
            while 0 <= k <= j_max:
                if used(k) != c:
                    return k
                k += d
            return None

        best = schedule(j0)
        # the better of the two neighbours, if it beats j0 strictly, gives
        # the direction; then on from neighbour to neighbour while it keeps
        # improving strictly
        near = [schedule(j) for j in (neighbour(j0, -1), neighbour(j0, 1)) if j is not None]
        if near and min(near, key=lambda c: c[0])[0] < best[0]:
            best = min(near, key=lambda c: c[0])
            step_dir = 1 if best[1] > j0 else -1
            j = neighbour(best[1], step_dir)
            while j is not None:
                cand = schedule(j)
                if cand[0] >= best[0]:
                    break
                best = cand
                j = neighbour(j, step_dir)
    if best is None:
        return CascadePlan(0, 0, 0, 0, [0] * (n_cta + 1), [], [], [0], [])
    (span, _), _, (_, q_pre, block_chunk, n_pre), (c_s, _, q_suf) = best
    np_block = [_ceil_div(l, c) for l, c in zip(block_lens, block_chunk)]
    units, merge_indptr = [], [0]
    for r in range(batch):
        n = np_block[block_of[r]] + _ceil_div(suf_len[r], c_s)
        units.append((r, n))
        merge_indptr.append(merge_indptr[-1] + n)
    p_ip = [int(x) for x in p_ip]
    s_ip = [int(x) for x in s_ip]
    nnz_p = p_ip[-1] if p_ip else 0
    cta_indptr, items = [0], []
    for q in q_pre:
        for cost, u, k, tb, te in q:
            b, head = divmod(u, hkv)
            r0, n, j = blocks[b]
            items.append((r0, tb, te, k, p_ip[j] + tb // P, n, -1, head))
        cta_indptr.append(len(items))
    for q in q_suf:
        for cost, r, k, tb, te in q:
            items.append((r, tb, te, merge_indptr[r] + np_block[block_of[r]] + k,
                          nnz_p + s_ip[r] + tb // P, 1, 0, 0))
        cta_indptr.append(len(items))
    page_list = [int(x) for x in p_ix[:nnz_p]] + [int(x) for x in s_ix[:s_ip[-1] if s_ip else 0]]
    chunk_pre = max((min(c, l) for c, l in zip(block_chunk, block_lens)), default=0)
    return CascadePlan(n_pre, chunk_pre, c_s, span // 16, cta_indptr, items, units,
                       merge_indptr, page_list)
