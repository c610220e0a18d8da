"""Seeded synthetic inputs for paged-KV decode attention.

This module only *makes inputs*: request lengths, the CSR page table an
engine would hand to the planner, page placement in the pool, and the bf16
query / KV values.  It holds none of the attention arithmetic, and it is the
one module that both the CPU oracle (tests) and the CUDA path (tests, bench)
draw their inputs from.

Shapes and distributions follow the workloads named on the pages:

* worked example -- lengths [37, 16, 5], page size 16
  ("FlashInfer, in depth", section "The block-sparse page table");
* a Llama-3-8B-shaped step -- 32 layers, 32 query heads, 8 KV heads, head
  dim 128, bf16, 64 requests averaging ~4,000 tokens
  ("FlashInfer, in depth", section "Why serving attention is a different
  problem");
* 63 short requests plus one 100,000-token request
  ("FlashInfer, in depth", section "Load balancing with split-KV");
* a shared prefix plus per-request suffixes
  ("FlashInfer 完全拆解", section "Composable Format");
* page size 1, token-level sparse layout
  ("FlashInfer, in depth", section "The block-sparse page table");
* the Llama-shaped step with an E4M3 cache, and either step with the cache in
  the HND layout [pages, 2, Hkv, P, D] ("FlashInfer 完全拆解", section
  接口层最容易踩的四个坑) -- the same values as the NHD cache, moved.

Values are N(0, 1) in bf16.  Pages are placed by a seeded permutation of the
pool, so consecutive logical pages are scattered in memory.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

__all__ = [
    "Workload",
    "WORKLOADS",
    "page_table",
    "make_tables",
    "make_q",
    "make_kv",
    "make_kv_fp8",
    "workload",
]


@dataclass(frozen=True)
class Workload:
    """One synthetic decode workload (shapes + seeded length recipe)."""

    name: str
    seed: int
    hq: int
    hkv: int
    head_dim: int
    page_size: int
    layers: int
    lens: tuple  # per-request KV lengths (tokens)
    pool_pages: int  # pages in the pool (>= pages referenced)
    prefix_tokens: int = 0  # shared-prefix workload only
    suffix_lens: tuple = field(default_factory=tuple)
    kv_dtype: str = "bf16"  # "bf16" or "e4m3" (FP8 cache with K / V scales)
    kv_layout: str = "NHD"  # "NHD" [pages, 2, P, Hkv, D] or "HND" [pages, 2, Hkv, P, D]

    @property
    def kv_elem_bytes(self) -> int:
        return 1 if self.kv_dtype == "e4m3" else 2

    @property
    def batch(self) -> int:
        return len(self.lens)


def _randint(gen: torch.Generator, lo: int, hi: int, n: int) -> list:
    """n integers uniform in [lo, hi] (inclusive), from a seeded CPU generator."""
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


def _pages_for(lens, page_size) -> int:
    return sum(int(math.ceil(n / page_size)) for n in lens)


def workload(name: str) -> Workload:
    """Build the named workload.  Lengths are drawn from torch's CPU
    generator seeded with the workload's seed, so they are the same on any
    machine."""
    if name == "worked_example":
        lens = (37, 16, 5)
        return Workload(name, 1, 32, 8, 128, 16, 1, lens, pool_pages=64)
    if name == "llama8b_step":
        g = torch.Generator().manual_seed(2)
        lens = tuple(_randint(g, 1, 8192, 64))
        return Workload(name, 2, 32, 8, 128, 16, 32, lens, _pages_for(lens, 16))
    if name in ("llama8b_step_fp8", "llama8b_step_hnd", "llama8b_step_fp8_hnd"):
        w = workload("llama8b_step")
        return Workload(name, w.seed, w.hq, w.hkv, w.head_dim, w.page_size, w.layers, w.lens,
                        w.pool_pages, kv_dtype="e4m3" if "fp8" in name else "bf16",
                        kv_layout="HND" if name.endswith("hnd") else "NHD")
    if name == "skewed":
        g = torch.Generator().manual_seed(3)
        lens = tuple(_randint(g, 128, 512, 63) + [100_000])
        return Workload(name, 3, 32, 8, 128, 16, 1, lens, _pages_for(lens, 16))
    if name == "shared_prefix_hnd":
        w = workload("shared_prefix")
        return Workload(name, w.seed, w.hq, w.hkv, w.head_dim, w.page_size, w.layers, w.lens,
                        w.pool_pages, prefix_tokens=w.prefix_tokens, suffix_lens=w.suffix_lens,
                        kv_layout="HND")
    if name == "shared_prefix":
        g = torch.Generator().manual_seed(4)
        suffix = tuple(_randint(g, 64, 1024, 32))
        prefix = 8192
        lens = tuple(prefix + s for s in suffix)
        pool = prefix // 16 + _pages_for(suffix, 16)
        return Workload(name, 4, 32, 8, 128, 16, 1, lens, pool,
                        prefix_tokens=prefix, suffix_lens=suffix)
    if name.startswith("prefix_") and "_b" in name:   # prefix_<tokens>_b<batch>
        prefix, batch = name[len("prefix_"):].split("_b")
        return shared_prefix_case(int(prefix), int(batch))
    if name == "token_sparse":
        g = torch.Generator().manual_seed(5)
        lens = tuple(_randint(g, 512, 2048, 512))
        return Workload(name, 5, 64, 8, 128, 1, 1, lens, sum(lens))
    raise KeyError(name)


WORKLOADS = ("worked_example", "llama8b_step", "skewed", "shared_prefix", "token_sparse")
# the same Llama-shaped step over an E4M3 cache
EXTRA_WORKLOADS = ("llama8b_step_fp8", "llama8b_step_hnd", "llama8b_step_fp8_hnd",
                   "shared_prefix_hnd")


def page_table(kv_lens, page_size, page_ids=None):
    """CSR page metadata an engine builds from per-request KV lengths.

    Request i gets ceil(l_i / P) pages, taken in order from ``page_ids``
    (default: 0, 1, 2, ...); its last page holds l_i - (pages - 1) * P
    tokens, a value in 1..P.  Returns int32 numpy arrays
    (indptr[B+1], indices[nnz], last_page_len[B]).
    """
    indptr = [0]
    last = []
    n_pages = []
    for n in kv_lens:
        if n < 1:
            raise ValueError("a request needs at least one token")
        pages = -(-int(n) // page_size)
        n_pages.append(pages)
        indptr.append(indptr[-1] + pages)
        last.append(int(n) - (pages - 1) * page_size)
    nnz = indptr[-1]
    if page_ids is None:
        indices = np.arange(nnz, dtype=np.int32)
    else:
        indices = np.asarray(page_ids[:nnz], dtype=np.int32)
        if indices.shape[0] != nnz:
            raise ValueError("not enough page ids")
    return (np.asarray(indptr, dtype=np.int32), indices,
            np.asarray(last, dtype=np.int32))


def _perm(seed: int, n: int) -> np.ndarray:
    g = torch.Generator().manual_seed(1000 + seed)
    return torch.randperm(n, generator=g).numpy().astype(np.int32)


def shared_prefix_case(prefix: int, batch: int, suffix: int = 128) -> Workload:
    """A batch of `batch` requests sharing a `prefix`-token prefix, each with
    its own `suffix`-token tail (page size 16, Hq 32 / Hkv 8, D 128): the
    shape of the Composable Format latency table (FlashInfer 完全拆解,
    Composable Format 只在复用足够大时占优: suffix 128, batch 16 and 64,
    prefix 1,024 / 8,192 / 32,768)."""
    suffix_lens = tuple([suffix] * batch)
    lens = tuple(prefix + s for s in suffix_lens)
    pool = prefix // 16 + _pages_for(suffix_lens, 16)
    return Workload(f"prefix_{prefix}_b{batch}", 6, 32, 8, 128, 16, 1, lens, pool,
                    prefix_tokens=prefix, suffix_lens=suffix_lens)


def make_tables(w: Workload):
    """Page tables for a workload, with pages scattered over the pool.

    Returns a dict.  For every workload: ``indptr``, ``indices``, ``last``
    (the full-length view).  For the shared-prefix workload also
    ``prefix`` and ``suffix``: (indptr, indices, last) views whose union is
    the full view -- every request's prefix rows point at the same pages.
    """
    perm = _perm(w.seed, w.pool_pages)
    out = {}
    if w.prefix_tokens:
        P = w.page_size
        n_pre = w.prefix_tokens // P
        pre_pages = perm[:n_pre]
        suf_ids = perm[n_pre:]
        s_indptr, s_indices, s_last = page_table(w.suffix_lens, P, suf_ids)
        B = w.batch
        p_indptr = np.arange(B + 1, dtype=np.int32) * n_pre
        p_indices = np.tile(pre_pages, B).astype(np.int32)
        p_last = np.full(B, P, dtype=np.int32)
        out["prefix"] = (p_indptr, p_indices, p_last)
        out["suffix"] = (s_indptr, s_indices, s_last)
        # full view: prefix pages then the request's own suffix pages
        rows = []
        for i in range(B):
            rows.append(np.concatenate([pre_pages,
                                        s_indices[s_indptr[i]:s_indptr[i + 1]]]))
        indptr = np.zeros(B + 1, dtype=np.int32)
        indptr[1:] = np.cumsum([len(r) for r in rows])
        out["indptr"] = indptr
        out["indices"] = np.concatenate(rows).astype(np.int32)
        out["last"] = s_last.copy()
    else:
        out["indptr"], out["indices"], out["last"] = page_table(
            w.lens, w.page_size, perm)
    return out


def _generator(seed: int, device) -> torch.Generator:
    return torch.Generator(device=device).manual_seed(seed)


def make_q(w: Workload, device="cpu", layers=None, seed_offset=0):
    """bf16 queries ~ N(0, 1): list (one per layer) of [B, Hq, D] tensors."""
    layers = w.layers if layers is None else layers
    g = _generator(10_000 * w.seed + 17 + seed_offset, device)
    return [torch.randn(w.batch, w.hq, w.head_dim, generator=g,
                        dtype=torch.bfloat16, device=device)
            for _ in range(layers)]


def _layout(x, w: Workload):
    """An NHD cache in the workload's layout (HND: heads before slots)."""
    return x.permute(0, 1, 3, 2, 4).contiguous() if w.kv_layout == "HND" else x


def make_kv(w: Workload, device="cpu", layers=None, seed_offset=0):
    """bf16 paged caches ~ N(0, 1): list (one per layer) of NHD tensors
    [pool_pages, 2, P, Hkv, D] (K at index 0 of dim 1, V at index 1), or the
    same values as HND [pool_pages, 2, Hkv, P, D] for an HND workload."""
    layers = w.layers if layers is None else layers
    g = _generator(10_000 * w.seed + 29 + seed_offset, device)
    shape = (w.pool_pages, 2, w.page_size, w.hkv, w.head_dim)
    return [_layout(torch.randn(shape, generator=g, dtype=torch.bfloat16, device=device), w)
            for _ in range(layers)]


FP8_AMAX = 4.0   # N(0, 1) values are clipped to +-4 (the E4M3 maximum 448 after scaling)


def make_kv_fp8(w: Workload, device="cpu", layers=None, seed_offset=0, amax=FP8_AMAX):
    """E4M3 paged caches (torch.float8_e4m3fn, NHD) holding N(0, 1) / scale
    values, scale = amax / 448 so that amax maps to the largest E4M3 value;
    returns (caches, scale) -- the attended K and V are scale * cache."""
    layers = w.layers if layers is None else layers
    scale = amax / 448.0
    g = _generator(10_000 * w.seed + 31 + seed_offset, device)
    shape = (w.pool_pages, 2, w.page_size, w.hkv, w.head_dim)
    caches = []
    for _ in range(layers):
        x = torch.randn(shape, generator=g, dtype=torch.bfloat16, device=device)
        caches.append(_layout((x.float() / scale).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn),
                              w))
    return caches, scale


def random_small(seed: int, batch: int, max_len: int, page_size: int,
                 hq: int = 8, hkv: int = 2, head_dim: int = 128,
                 min_len: int = 1, extra_pages: int = 3):
    """A small random workload for tests: lengths uniform in
    [min_len, max_len], pages scattered over a pool with a few unused pages."""
    g = torch.Generator().manual_seed(50_000 + seed)
    lens = tuple(_randint(g, min_len, max_len, batch))
    pool = _pages_for(lens, page_size) + extra_pages
    return Workload(f"random{seed}", 100 + seed, hq, hkv, head_dim, page_size,
                    1, lens, pool)
