"""CPU-only checks of the C-ABI library: it builds, loads, exports every
entry point its header declares, and its host scheduler matches the plan
restatement integer for integer.  No GPU work is issued here."""
import ctypes
import os
import re

import numpy as np
import pytest

import paged_kv_decode_host_gb300 as pkd
import workloads
from oracle import plan as oplan

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pkd.build()
    return pkd.load()


def _declared():
    names = set()
    with open(os.path.join(ROOT, "include", "pkd.h")) as f:
        text = f.read()
    for m in re.finditer(r"\b(pkd_[a-z_]+)\s*\(", text):
        names.add(m.group(1))
    return names


def test_exports_every_declared_symbol(lib):
    declared = _declared()
    assert declared, "no declarations parsed"
    assert declared == set(pkd.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name
    assert lib.pkd_version() >= 100
    assert lib.pkd_status_str(-2).decode().startswith("bad page table")
    assert lib.pkd_status_str(12345).decode() == "unknown status"


def _cfg(P, hq=32, hkv=8, max_batch=64, max_pages=4096, num_pages=4096, n_cta=152,
         alpha=-1, min_chunk=-1, d=128):
    return pkd.make_config(hq, hkv, d, P, max_batch, max_pages, num_pages, alpha, min_chunk,
                           n_cta)


def test_config_validation(lib):
    off = (ctypes.c_int64 * 6)()
    bad = [
        _cfg(16, d=64),                 # head dim other than 128
        _cfg(16, hq=12, hkv=8),         # Hq % Hkv != 0
        _cfg(16, hq=48, hkv=8),         # group of 6
        _cfg(16, hq=32, hkv=16),        # more than 8 KV heads
    ]
    for c in bad:
        assert lib.pkd_schedule_layout(ctypes.byref(c), off) == -3
    for bad_flags in (3, 5, 7, 9, 12, 28, 33 | 4 | 8, 128, 512, 256 | 1, 256 | 4, 256 | 8,
                      256 | 16, 256 | 64, 256 | 128, 0x80000000):
        c = _cfg(16)
        c.flags = bad_flags
        assert lib.pkd_schedule_layout(ctypes.byref(c), off) == -1
    for ok_flags in (0, 1, 2, 4, 6, 8, 10, 16, 17, 18, 20, 24, 32, 33, 36, 40, 56, 64, 65, 66,
                     68, 72, 88, 120, 256, 256 | 2, 256 | 32, 256 | 34):
        c = _cfg(16)
        c.flags = ok_flags
        assert lib.pkd_schedule_layout(ctypes.byref(c), off) == 0
    assert lib.pkd_schedule_layout(ctypes.byref(_cfg(16)), off) == 0
    assert list(off)[5] > list(off)[4] > list(off)[3] > list(off)[2] > list(off)[1] > list(off)[0]


def _compare(cfg, indptr, indices, last, alpha, min_chunk, chunk_rule="closed"):
    words, info, off = pkd.plan_host(cfg, indptr, indices, last)
    got = pkd.decode_schedule(words, off, info)
    ref = oplan.plan(indptr, indices, last, page_size=cfg.page_size, num_pages=cfg.num_pages,
                     n_cta=cfg.num_ctas, alpha=alpha, min_chunk_tokens=min_chunk,
                     chunk_rule=chunk_rule)
    # header word 16: the most chunks of any split request
    assert got["header"][16] == max([n for _, n in ref.units], default=0)
    assert got["header"][17:19] == [cfg.max_batch, cfg.max_num_pages]
    assert got["header"][19:] == [0] * 13
    assert info["chunk_tokens"] == ref.chunk
    assert info["makespan"] == ref.makespan
    assert info["num_items"] == ref.n_items
    assert info["num_slots"] == ref.n_slots
    assert got["cta_indptr"] == ref.cta_indptr
    assert got["items"] == [tuple(x) for x in ref.items]
    assert got["units"] == [tuple(x) for x in ref.units]
    assert got["merge_indptr"] == ref.merge_indptr
    assert got["page_list"] == ref.page_list
    assert got["header"][0] == 0x31444B50
    return info


@pytest.mark.parametrize("name", ["worked_example", "llama8b_step", "skewed",
                                  "shared_prefix", "token_sparse"])
def test_plan_bit_exact_on_workloads(lib, name):
    w = workloads.workload(name)
    t = workloads.make_tables(w)
    views = [(t["indptr"], t["indices"], t["last"])]
    if "prefix" in t:
        views += [t["prefix"], t["suffix"]]
    for indptr, indices, last in views:
        nnz = int(indptr[-1])
        cfg = _cfg(w.page_size, w.hq, w.hkv, max_batch=w.batch, max_pages=nnz,
                   num_pages=w.pool_pages, n_cta=152, alpha=32, min_chunk=256)
        _compare(cfg, indptr, indices, last, 32, 256)


@pytest.mark.parametrize("seed", range(12))
def test_plan_bit_exact_random(lib, seed):
    rng = np.random.default_rng(100 + seed)
    P = int(rng.choice([1, 2, 3, 8, 16, 32]))
    B = int(rng.integers(0 if seed == 0 else 1, 70))
    lens = rng.integers(1, 5000, B).tolist()
    if seed % 3 == 1 and B:
        lens[-1] = int(rng.integers(20000, 120000))
    pool = sum(-(-l // P) for l in lens) + 7
    ids = rng.permutation(pool).astype(np.int32)
    indptr, indices, last = workloads.page_table(lens, P, ids)
    n_cta = int(rng.choice([1, 7, 64, 152, 304]))
    alpha = int(rng.integers(0, 200))
    min_chunk = int(rng.choice([1, 16, 256, 1000]))
    cfg = _cfg(P, max_batch=max(B, 1), max_pages=max(int(indptr[-1]), 1), num_pages=pool,
               n_cta=n_cta, alpha=alpha, min_chunk=min_chunk)
    info = _compare(cfg, indptr, indices, last, alpha, min_chunk)
    assert info["batch"] == B


@pytest.mark.parametrize("seed", range(10))
def test_search_rule_plan_bit_exact_random(lib, seed):
    """Binary-search chunk rule (PKD_FLAG_CHUNK_SEARCH) against the oracle's
    scan, schedule word for word."""
    rng = np.random.default_rng(300 + seed)
    P = int(rng.choice([1, 3, 16, 32]))
    B = int(rng.integers(0 if seed == 0 else 1, 300))
    lens = rng.integers(1, 6000, B).tolist()
    if seed % 3 == 1 and B:
        lens[-1] = int(rng.integers(20000, 120000))
    pool = sum(-(-l // P) for l in lens) + 7
    indptr, indices, last = workloads.page_table(lens, P, rng.permutation(pool).astype(np.int32))
    n_cta = int(rng.choice([1, 7, 64, 152, 304]))
    alpha = int(rng.integers(0, 200))
    min_chunk = int(rng.choice([1, 16, 256, 1000]))
    cfg = _cfg(P, max_batch=max(B, 1), max_pages=max(int(indptr[-1]), 1), num_pages=pool,
               n_cta=n_cta, alpha=alpha, min_chunk=min_chunk)
    cfg.flags = pkd.FLAG_CHUNK_SEARCH
    _compare(cfg, indptr, indices, last, alpha, min_chunk, chunk_rule="search")


@pytest.mark.parametrize("name", ["llama8b_step", "skewed", "token_sparse"])
def test_search_rule_plan_bit_exact_on_workloads(lib, name):
    w = workloads.workload(name)
    t = workloads.make_tables(w)
    nnz = int(t["indptr"][-1])
    cfg = _cfg(w.page_size, w.hq, w.hkv, max_batch=w.batch, max_pages=nnz,
               num_pages=w.pool_pages, n_cta=152, alpha=32, min_chunk=256)
    cfg.flags = pkd.FLAG_CHUNK_SEARCH
    _compare(cfg, t["indptr"], t["indices"], t["last"], 32, 256, chunk_rule="search")


def test_plan_host_rejects_bad_tables(lib):
    cfg = _cfg(16, max_batch=4, max_pages=8, num_pages=8, n_cta=4)
    cases = [
        ([0, 2], [0, 1], [0]),           # last_page_len 0 (multiple-of-P bug)
        ([0, 2], [0, 1], [17]),          # longer than the page
        ([0, 0], [], [1]),               # empty request
        ([0, 1], [8], [1]),              # page outside the pool
        ([0, 1], [-3], [1]),             # negative page
        ([1, 2], [0, 1], [1]),           # indptr[0] != 0
    ]
    for indptr, indices, last in cases:
        with pytest.raises(pkd.PkdError) as e:
            pkd.plan_host(cfg, np.array(indptr, np.int32), np.array(indices, np.int32),
                          np.array(last, np.int32))
        assert e.value.status == -2, (indptr, indices, last)
    # capacity: batch above max_batch, pages above max_num_pages
    with pytest.raises(pkd.PkdError) as e:
        pkd.plan_host(cfg, np.arange(6, dtype=np.int32), np.arange(5, dtype=np.int32),
                      np.ones(5, np.int32))
    assert e.value.status == -7
    with pytest.raises(pkd.PkdError) as e:
        pkd.plan_host(cfg, np.array([0, 9], np.int32), np.zeros(9, np.int32),
                      np.ones(1, np.int32))
    assert e.value.status == -7
    # int64 tables are refused by the binding before reaching the library
    with pytest.raises(TypeError):
        pkd.plan_host(cfg, np.array([0, 1]), np.array([0]), np.array([1]))


@pytest.mark.parametrize("seed", range(8))
def test_grouped_plan_bit_exact_random(lib, seed):
    rng = np.random.default_rng(300 + seed)
    P = int(rng.choice([1, 3, 16]))
    hkv = 8
    g = int(rng.choice([1, 2, 4, 8]))
    n_groups = int(rng.integers(1, 5))
    sizes = rng.integers(1, 35, n_groups).tolist()
    group_indptr = np.array([0] + np.cumsum(sizes).tolist(), dtype=np.int32)
    lens = rng.integers(1, 12000, n_groups).tolist()
    pool = sum(-(-l // P) for l in lens) + 4
    indptr, indices, last = workloads.page_table(lens, P, rng.permutation(pool).astype(np.int32))
    n_cta = int(rng.choice([3, 64, 152]))
    cfg = pkd.make_config(g * hkv, hkv, 128, P, int(group_indptr[-1]), int(indptr[-1]), pool,
                          32, 256, n_cta, pkd.FLAG_SHARED_PREFIX)
    words, info, off = pkd.plan_host_shared(cfg, group_indptr, indptr, indices, last)
    got = pkd.decode_schedule(words, off, info)
    ref = oplan.plan(indptr, indices, last, page_size=P, num_pages=pool, n_cta=n_cta, alpha=32,
                     min_chunk_tokens=256, group_indptr=group_indptr, rows=16 // g)
    assert info["chunk_tokens"] == ref.chunk and info["makespan"] == ref.makespan
    assert got["cta_indptr"] == ref.cta_indptr
    assert got["items"] == [tuple(x) for x in ref.items]
    assert got["units"] == [tuple(x) for x in ref.units]
    assert got["merge_indptr"] == ref.merge_indptr
    assert got["page_list"] == ref.page_list
    assert got["header"][15] == 16 // g


@pytest.mark.parametrize("seed", range(8))
def test_dense_prefix_plan_bit_exact_random(lib, seed):
    """Dense-prefix plans (blocks of 128 / g requests, one KV head per work
    item) against the oracle's per-head restatement, word for word; every
    (request, head, token) covered exactly once."""
    rng = np.random.default_rng(700 + seed)
    P = int(rng.choice([16, 32, 64]))
    hkv = int(rng.choice([1, 2, 8]))
    g = int(rng.choice([1, 2, 4, 8]))
    n_groups = int(rng.integers(1, 4))
    sizes = rng.integers(1, 300, n_groups).tolist()
    group_indptr = np.array([0] + np.cumsum(sizes).tolist(), dtype=np.int32)
    lens = rng.integers(1, 12000, n_groups).tolist()
    pool = sum(-(-l // P) for l in lens) + 4
    indptr, indices, last = workloads.page_table(lens, P, rng.permutation(pool).astype(np.int32))
    n_cta = int(rng.choice([3, 64, 152]))
    flags = pkd.FLAG_SHARED_PREFIX | pkd.FLAG_DENSE_PREFIX
    rule = "closed"
    if seed % 3 == 2:
        flags |= pkd.FLAG_CHUNK_SEARCH
        rule = "search"
    cfg = pkd.make_config(g * hkv, hkv, 128, P, int(group_indptr[-1]), int(indptr[-1]), pool,
                          32, 256, n_cta, flags)
    words, info, off = pkd.plan_host_shared(cfg, group_indptr, indptr, indices, last)
    got = pkd.decode_schedule(words, off, info)
    ref = oplan.plan(indptr, indices, last, page_size=P, num_pages=pool, n_cta=n_cta, alpha=32,
                     min_chunk_tokens=256, group_indptr=group_indptr, rows=128 // g,
                     chunk_rule=rule, per_head=hkv)
    assert info["chunk_tokens"] == ref.chunk and info["makespan"] == ref.makespan
    assert got["cta_indptr"] == ref.cta_indptr
    assert got["items"] == [tuple(x) for x in ref.items]
    assert got["heads"] == ref.heads
    assert got["units"] == [tuple(x) for x in ref.units]
    assert got["merge_indptr"] == ref.merge_indptr
    assert got["header"][15] == 128 // g
    assert info["total_tokens"] == sum(ref.lens)
    # coverage per head: each (request, head, token) exactly once
    req_row = [j for j in range(len(lens)) for _ in range(sizes[j])]
    seen = {}
    for (r0, tb, te, dst, fp, n, stride), hd in zip(got["items"], got["heads"]):
        assert 0 <= hd < hkv and n <= 128 // g
        for r in range(r0, r0 + n):
            a = seen.setdefault((r, hd), np.zeros(lens[req_row[r]], np.int32))
            a[tb:te] += 1
    assert len(seen) == len(req_row) * hkv
    assert all(np.all(a == 1) for a in seen.values())


def test_plan_fast_path_marshalling():
    """The compiled plan fast path hands the C ABI the arrays' own buffers,
    the batch and the stream, returns the entry point's status and epoch, and
    leaves every input it cannot pass as-is (int64, lists, short or
    non-contiguous arrays) to the general path (status 1000).  Checked on
    the CPU against a stand-in entry point; the real ones are restored."""
    import ctypes
    m = pytest.importorskip("paged_kv_decode_host_gb300._pkd_plan")
    lib = pkd.load()
    calls = []
    plan_t = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                              ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                              ctypes.POINTER(ctypes.c_uint64))
    shared_t = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint64))

    def fake_plan(ctx, ip, ix, la, batch, stream, ep):
        calls.append(("plan", ctx, ip, ix, la, batch, stream))
        ep[0] = 41
        return -2 if batch == 3 else 0

    def fake_shared(ctx, gi, ng, ip, ix, la, stream, ep):
        calls.append(("shared", ctx, gi, ng, ip, ix, la, stream))
        ep[0] = 42
        return 0

    vp = ctypes.c_void_p
    cascade_t = ctypes.CFUNCTYPE(ctypes.c_int, vp, vp, ctypes.c_int32, vp, vp, vp, vp, vp, vp, vp,
                                 ctypes.POINTER(ctypes.c_uint64))

    def fake_cascade(ctx, gi, ng, pip, pix, pla, sip, six, sla, stream, ep):
        calls.append(("cascade", ctx, gi, ng, pip, pix, pla, sip, six, sla, stream))
        ep[0] = 43
        return 0

    cb_plan, cb_shared = plan_t(fake_plan), shared_t(fake_shared)
    cb_cascade = cascade_t(fake_cascade)
    try:
        m.init(ctypes.cast(cb_plan, ctypes.c_void_p).value,
               ctypes.cast(cb_shared, ctypes.c_void_p).value,
               ctypes.cast(cb_cascade, ctypes.c_void_p).value)
        ip = np.array([0, 3, 4], np.int32)
        ix = np.arange(4, dtype=np.int32)
        la = np.array([5, 16], np.int32)
        assert m.plan(123, ip, ix, la, 456) == (0, 41)
        assert calls[-1] == ("plan", 123, ip.ctypes.data, ix.ctypes.data, la.ctypes.data, 2, 456)
        ip3, la3 = np.array([0, 1, 2, 4], np.int32), np.array([1, 1, 1], np.int32)
        assert m.plan(1, ip3, ix, la3, 0)[0] == -2          # the entry point's status
        n = len(calls)
        for args in ((ip.astype(np.int64), ix, la), ([0, 3, 4], ix, la), (ip, ix[:2], la),
                     (ip[:2], ix, la), (np.zeros(6, np.int32)[::2], ix, la)):
            assert m.plan(1, *args, 0)[0] == 1000
        assert len(calls) == n                               # none reached the entry point
        gi = np.array([0, 32], np.int32)
        assert m.plan_shared(7, gi, np.array([0, 4], np.int32), ix, np.array([16], np.int32),
                             9) == (0, 42)
        assert calls[-1][0] == "shared" and calls[-1][3] == 1 and calls[-1][7] == 9
        assert m.plan_shared(7, gi, ip, ix, la, 9)[0] == 1000   # groups mismatch
        # cascade: one group of 2 requests over 4 prefix pages, suffixes of 3 and 1 pages
        g2 = np.array([0, 2], np.int32)
        pre = (np.array([0, 4], np.int32), ix, np.array([16], np.int32))
        suf = (ip, ix, la)
        assert m.plan_cascade(5, g2, *pre, *suf, 8) == (0, 43)
        assert calls[-1] == ("cascade", 5, g2.ctypes.data, 1, pre[0].ctypes.data,
                             ix.ctypes.data, pre[2].ctypes.data, ip.ctypes.data, ix.ctypes.data,
                             la.ctypes.data, 8)
        n = len(calls)
        for bad in ((np.array([0, 3], np.int32), *pre, *suf),           # group size != batch
                    (g2, *pre, ip.astype(np.int64), ix, la),             # int64 suffix indptr
                    (g2, pre[0], ix[:3], pre[2], *suf),                  # prefix indices short
                    (g2, *pre, ip, ix[:3], la)):                         # suffix indices short
            assert m.plan_cascade(5, *bad, 8)[0] == 1000
        assert len(calls) == n
    finally:
        m.init(ctypes.cast(lib.pkd_plan, ctypes.c_void_p).value,
               ctypes.cast(lib.pkd_plan_shared, ctypes.c_void_p).value,
               ctypes.cast(lib.pkd_plan_cascade, ctypes.c_void_p).value)


def test_static_scratch_rejects_mismatched_schedules(lib):
    """pkd_run_static_scratch checks a host schedule against the layout of the
    configuration it is given before anything reaches the GPU: a schedule
    planned for other capacities (other word offsets) or with an index out of
    range is refused with INVALID_ARG, no CUDA call made."""
    import torch
    if torch.cuda.is_available():
        # stand-in device pointers below: never let a schedule that the check
        # should refuse reach a real GPU
        pytest.skip("host-only check; runs where no GPU is present")
    w = workloads.workload("skewed")
    t = workloads.make_tables(w)
    nnz = int(t["indptr"][-1])
    cfg = pkd.make_config(w.hq, w.hkv, 128, 16, w.batch, nnz, w.pool_pages, -1, -1, 152)
    words, info, off = pkd.plan_host(cfg, t["indptr"], t["indices"], t["last"])
    fake = ctypes.c_void_p(1 << 12)   # aligned, non-null: only the schedule decides

    def run(c, wd):
        return lib.pkd_run_static_scratch(ctypes.byref(c), ctypes.c_void_p(wd.ctypes.data),
                                          wd.size, fake, fake, fake, fake, None)

    # the untouched schedule passes every host check and only then needs the
    # device (none here: a CUDA error, not INVALID_ARG)
    assert run(cfg, words) == -8

    for field, delta in (("max_batch", 1), ("max_num_pages", 16)):
        other = pkd.make_config(w.hq, w.hkv, 128, 16, w.batch, nnz, w.pool_pages, -1, -1, 152)
        setattr(other, field, getattr(other, field) + delta)
        # planned for cfg, run against a layout with other offsets
        assert run(other, np.resize(words, pkd.schedule_layout(other)[5])) == -1
    corrupt = []
    item0 = off[1]
    bad = words.copy()
    bad[item0 + 3] = 10 ** 6                      # partial-state slot past the layout
    corrupt.append(bad)
    bad = words.copy()
    bad[item0 + 4] = nnz                          # first page past the page list
    corrupt.append(bad)
    bad = words.copy()
    bad[item0 + 0] = w.batch                      # request outside the batch
    corrupt.append(bad)
    bad = words.copy()
    bad[off[0] + 1] = bad[off[0] + 2] + 1         # CTA queues out of order
    corrupt.append(bad)
    bad = words.copy()
    bad[off[3] + 1] = 10 ** 6                     # merge range past the slots
    corrupt.append(bad)
    for bad in corrupt:
        assert run(cfg, bad) == -1


def _cascade_cfg(hq, hkv, batch, nnz, pool, n_cta, flags=0):
    return pkd.make_config(hq, hkv, 128, 16, batch, nnz, pool, -1, -1, n_cta,
                           pkd.FLAG_CASCADE | flags)


def _compare_cascade(cfg, gi, prefix, suffix):
    words, info, off = pkd.plan_host_cascade(cfg, gi, prefix, suffix)
    g = cfg.num_qo_heads // cfg.num_kv_heads
    ref = oplan.plan_cascade(gi, prefix, suffix, page_size=16, num_pages=cfg.num_pages,
                             n_cta=cfg.num_ctas, hkv=cfg.num_kv_heads, rows=128 // g, alpha=32,
                             prefix_alpha=512, prefix_cost16=3, suffix_floor=128)
    got = pkd.decode_schedule(words, off, info)
    items = [tuple(int(x) for x in r)
             for r in words[off[1]:off[1] + 8 * info["num_items"]].reshape(-1, 8)]
    assert info["prefix_ctas"] == ref.n_pre == got["header"][19]
    assert info["prefix_chunk_tokens"] == ref.chunk_pre == got["header"][20]
    assert info["chunk_tokens"] == ref.chunk_suf
    assert info["makespan"] == ref.makespan
    assert got["cta_indptr"] == ref.cta_indptr
    assert items == ref.items
    assert got["units"] == [tuple(x) for x in ref.units]
    assert got["merge_indptr"] == ref.merge_indptr
    assert got["page_list"] == ref.page_list
    assert got["header"][16] == max((n for _, n in ref.units), default=0)
    return info


def test_cascade_plan_bit_exact_shared_prefix_workload(lib):
    w = workloads.workload("shared_prefix")
    t = workloads.make_tables(w)
    n_pre = w.prefix_tokens // 16
    prefix = (np.array([0, n_pre], np.int32), np.asarray(t["prefix"][1][:n_pre], np.int32),
              np.array([16], np.int32))
    cfg = _cascade_cfg(32, 8, w.batch, n_pre + int(t["suffix"][0][-1]), w.pool_pages, 152)
    info = _compare_cascade(cfg, np.array([0, w.batch], np.int32), prefix, t["suffix"])
    assert 1 <= info["prefix_ctas"] < 152


@pytest.mark.parametrize("seed", range(8))
def test_cascade_plan_bit_exact_random(lib, seed):
    rng = np.random.default_rng(300 + seed)
    n_groups = int(rng.integers(1, 5))
    sizes = rng.integers(1, 60, n_groups).tolist()
    gi = np.array([0] + np.cumsum(sizes).tolist(), np.int32)
    B = int(gi[-1])
    plens = rng.integers(1, 30000, n_groups).tolist()
    slens = rng.integers(1, 4000, B).tolist()
    n_pp = sum(-(-l // 16) for l in plens)
    n_sp = sum(-(-l // 16) for l in slens)
    pool = n_pp + n_sp + 7
    ids = rng.permutation(pool).astype(np.int32)
    prefix = workloads.page_table(plens, 16, ids[:n_pp])
    suffix = workloads.page_table(slens, 16, ids[n_pp:n_pp + n_sp])
    hq, hkv = [(32, 8), (64, 8), (16, 8), (8, 8), (8, 2)][seed % 5]
    n_cta = int(rng.choice([2, 40, 152]))
    cfg = _cascade_cfg(hq, hkv, B + int(rng.integers(0, 9)), n_pp + n_sp, pool, n_cta)
    _compare_cascade(cfg, gi, prefix, suffix)


def test_cascade_plan_errors(lib):
    prefix = workloads.page_table([100], 16)                       # pages 0..6
    suffix = workloads.page_table([5, 20], 16, np.array([7, 8, 9], np.int32))
    cfg = _cascade_cfg(32, 8, 2, 10, 10, 152)
    gi = np.array([0, 2], np.int32)
    words, info, off = pkd.plan_host_cascade(cfg, gi, prefix, suffix)
    assert info["batch"] == 2 and info["num_units"] == 2
    with pytest.raises(pkd.PkdError) as e:                        # group with no request
        pkd.plan_host_cascade(cfg, np.array([0, 0], np.int32), prefix,
                              workloads.page_table([], 16))
    assert e.value.status == -2
    bad = (suffix[0], suffix[1], np.array([5, 17], np.int32))      # last page length > P
    with pytest.raises(pkd.PkdError) as e:
        pkd.plan_host_cascade(cfg, gi, prefix, bad)
    assert e.value.status == -2
    small = _cascade_cfg(32, 8, 2, 9, 10, 152)                      # 10 pages > capacity 9
    with pytest.raises(pkd.PkdError) as e:
        pkd.plan_host_cascade(small, gi, prefix, suffix)
    assert e.value.status == -7
    out_of_pool = (suffix[0], np.array([7, 8, 10], np.int32), suffix[2])
    with pytest.raises(pkd.PkdError) as e:
        pkd.plan_host_cascade(cfg, gi, prefix, out_of_pool)
    assert e.value.status == -2
    with pytest.raises(pkd.PkdError) as e:                        # a plain plan on it
        pkd.plan_host(cfg, *suffix)
    assert e.value.status == -1
    for flags in (pkd.FLAG_SHARED_PREFIX, pkd.FLAG_KV_FP8, pkd.FLAG_FMA_CONSUMER,
                  pkd.FLAG_ROW_COPIES, pkd.FLAG_CHUNK_SEARCH):
        c = _cascade_cfg(32, 8, 2, 10, 10, 152, flags)
        assert lib.pkd_schedule_layout(ctypes.byref(c), (ctypes.c_int64 * 6)()) == -1
    c = pkd.make_config(32, 8, 128, 8, 2, 10, 10, -1, -1, 152, pkd.FLAG_CASCADE)   # P 8
    assert lib.pkd_schedule_layout(ctypes.byref(c), (ctypes.c_int64 * 6)()) == -3


def test_format_advice_matches_both_planners(lib):
    """pkd_advise_format predicts each format from its own planner: its
    cascade makespan is the cascade plan's, its single-format makespan the
    plain plan's over every request's whole table (prefix pages, then its
    own); the longer the shared prefix, the larger the predicted gain."""
    gains = []
    for prefix_tokens, batch in ((16, 64), (1024, 16), (8192, 16), (8192, 64), (32768, 64)):
        w = workloads.shared_prefix_case(prefix_tokens, batch)
        t = workloads.make_tables(w)
        n_pre = prefix_tokens // 16
        prefix = (np.array([0, n_pre], np.int32), np.asarray(t["prefix"][1][:n_pre], np.int32),
                  np.array([16], np.int32))
        gi = np.array([0, batch], np.int32)
        cfg = _cascade_cfg(32, 8, batch, n_pre + int(t["suffix"][0][-1]), w.pool_pages, 152)
        adv = pkd.advise_format(cfg, gi, prefix, t["suffix"])
        _, info, _ = pkd.plan_host_cascade(cfg, gi, prefix, t["suffix"])
        assert adv["cascade_makespan"] == info["makespan"]
        assert adv["prefix_ctas"] == info["prefix_ctas"]
        plain = pkd.make_config(32, 8, 128, 16, batch, int(t["indptr"][-1]), w.pool_pages, -1, -1,
                                152)
        _, pinfo, _ = pkd.plan_host(plain, t["indptr"], t["indices"], t["last"])
        assert adv["single_makespan"] == pinfo["makespan"]
        assert adv["use_cascade"] == int(adv["cascade_us"] < adv["single_us"])
        gains.append(adv["single_us"] / adv["cascade_us"])
    # a one-page prefix over 64 requests: no reuse to win (measured 13.35 us
    # cascade, 13.36 us single format on GB300)
    assert gains[0] < 1.0 < gains[1]
    assert gains == sorted(gains)
    with pytest.raises(pkd.PkdError):                  # a plain configuration is refused
        pkd.advise_format(pkd.make_config(32, 8, 128, 16, 16, 100, 100, -1, -1, 152),
                          np.array([0, 1], np.int32), workloads.page_table([16], 16),
                          workloads.page_table([5], 16))
