"""The allocation-free entry point, pkd_run_static_scratch.

It serves callers that may not allocate device memory (an engine whose
allocator owns the whole GPU, a process under a hard memory cap, a plugin
with no allocator): instead of a caller-provided workspace it keeps the
schedule and the split partial states in a static device array inside the
library.  Here it is called through the C ABI twice in a row -- the second
call on a different batch, so stale contents of the shared array from the
first call would show -- and each result is compared with the oracle and
with the regular entry point (pkd_run on a workspace) within the parity
tolerances used throughout the tests (2e-2 on bf16 outputs, 1e-3 on fp32
LSE).  The other cases cover the branches its decode kernel takes that the
skewed batch does not (page size 1 with group 8, the CUDA-core consumer,
four KV heads),
check that a warm call changes neither torch's allocations nor the device's
free memory, and read the device error word back through
pkd_static_scratch_last_error.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_host_gb300 as pkd
import workloads

pytestmark = pytest.mark.gpu

OUT_TOL = 2e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkd.build()
    pkd.load()


def _regular(w, tables, q, kv, n_cta, tc=None):
    ip, ix, la = tables
    dec = pkd.BatchDecodeWithPagedKVCache(w.hq, w.hkv, w.head_dim, w.page_size,
                                          max_batch=w.batch, max_num_pages=int(ip[-1]),
                                          num_pages=w.pool_pages, num_ctas=n_cta,
                                          use_tensor_cores=tc)
    dec.plan(ip, ix, la)
    out, lse = dec.run(q, kv)
    torch.cuda.synchronize()
    return out, lse, dec.plan_info()


def _call(cfg, words, q, kv, out, lse):
    return pkd.load().pkd_run_static_scratch(
        ctypes.byref(cfg), ctypes.c_void_p(words.ctypes.data), words.size,
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kv.data_ptr()),
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _static(cfg, tables, q, kv):
    words, info, off = pkd.plan_host(cfg, *tables)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((q.shape[0], q.shape[1]), float("nan"), dtype=torch.float32,
                     device=q.device)
    st = _call(cfg, words, q, kv, out, lse)
    assert st == 0, pkd.STATUS.get(st, st)
    torch.cuda.synchronize()
    return out, lse, info


def _last_error(cfg):
    v = ctypes.c_int32(-1)
    st = pkd.load().pkd_static_scratch_last_error(
        ctypes.byref(cfg), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
        ctypes.byref(v))
    assert st == 0, pkd.STATUS.get(st, st)
    return v.value


def _close(a_o, a_l, b_o, b_l):
    assert (a_o.float() - b_o.float()).abs().max().item() <= OUT_TOL
    assert (a_l - b_l).abs().max().item() <= LSE_TOL


def _against_oracle(w, tables, q, kv, out, lse):
    ref_o, ref_l = oracle.decode(q, kv, *tables, hq=w.hq, hkv=w.hkv)
    assert np.abs(out.double().cpu().numpy() - ref_o).max() <= OUT_TOL
    assert np.abs(lse.double().cpu().numpy() - ref_l).max() <= LSE_TOL


def test_static_scratch_matches_regular_path_twice():
    w = workloads.workload("skewed")          # 63 short + one 100k-token request
    t = workloads.make_tables(w)
    full = (t["indptr"], t["indices"], t["last"])
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    ref_o, ref_l, info = _regular(w, full, q, kv, n_cta=0)
    assert info["num_units"] >= 1                    # partial states are used
    n_cta = info["num_ctas"]
    cfg = pkd.make_config(w.hq, w.hkv, w.head_dim, w.page_size, w.batch,
                          int(t["indptr"][-1]), w.pool_pages, -1, -1, n_cta)

    # call 1: the full skewed batch
    o1, l1, i1 = _static(cfg, full, q, kv)
    assert i1["num_units"] == info["num_units"]
    _close(o1, l1, ref_o, ref_l)
    _against_oracle(w, full, q, kv, o1, l1)
    assert _last_error(cfg) == 0

    # call 2: another batch (the long request and 20 short ones, new q),
    # same configuration -- the array still holds call 1's contents
    keep = list(range(43, 64))
    lens = [w.lens[i] for i in keep]
    w2 = workloads.Workload("skewed_tail", 33, w.hq, w.hkv, w.head_dim, w.page_size, 1,
                            tuple(lens), w.pool_pages)
    t2 = workloads.make_tables(w2)
    tables2 = (t2["indptr"], t2["indices"], t2["last"])
    q2 = workloads.make_q(w2, device="cuda")[0]
    ref_o2, ref_l2, info2 = _regular(w2, tables2, q2, kv, n_cta=n_cta)
    assert info2["num_units"] >= 1
    o2, l2, _ = _static(cfg, tables2, q2, kv)
    _close(o2, l2, ref_o2, ref_l2)
    _against_oracle(w2, tables2, q2, kv, o2, l2)
    assert _last_error(cfg) == 0


def _token_sparse_small():
    """Page size 1, group 8 (Hq 64, Hkv 8), 48 requests of 512..2048 tokens,
    every token at its own pool slot: the token-sparse shape, scaled to fit
    the static array."""
    g = torch.Generator().manual_seed(55)
    lens = tuple(int(x) for x in torch.randint(512, 2049, (48,), generator=g))
    return workloads.Workload("ts_small", 55, 64, 8, 128, 1, 1, lens, sum(lens))


def _llama_like_small():
    g = torch.Generator().manual_seed(56)
    lens = tuple(int(x) for x in torch.randint(1, 3000, (24,), generator=g))
    return workloads.Workload("ll_small", 56, 32, 8, 128, 16, 1, lens,
                              sum(-(-n // 16) for n in lens))


def _four_kv_heads_small():
    """Hq 16 / Hkv 4 (four consumer warps instead of eight), page size 16,
    20 requests of 1..2,500 tokens."""
    g = torch.Generator().manual_seed(57)
    lens = tuple(int(x) for x in torch.randint(1, 2500, (20,), generator=g))
    return workloads.Workload("hkv4_small", 57, 16, 4, 128, 16, 1, lens,
                              sum(-(-n // 16) for n in lens) + 3)


@pytest.mark.parametrize("case", ["token_sparse_g8", "fma_consumer", "four_kv_heads"])
def test_static_scratch_other_branches(case):
    """Page size 1 with g = 8 (merged K|V copies), the CUDA-core consumer,
    and four KV heads: static against the oracle and the regular path,
    twice."""
    w = {"token_sparse_g8": _token_sparse_small, "fma_consumer": _llama_like_small,
         "four_kv_heads": _four_kv_heads_small}[case]()
    tc = False if case == "fma_consumer" else None
    flags = pkd.FLAG_FMA_CONSUMER if case == "fma_consumer" else 0
    t = workloads.make_tables(w)
    tables = (t["indptr"], t["indices"], t["last"])
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    ref_o, ref_l, info = _regular(w, tables, q, kv, n_cta=0, tc=tc)
    cfg = pkd.make_config(w.hq, w.hkv, w.head_dim, w.page_size, w.batch,
                          int(t["indptr"][-1]), w.pool_pages, -1, -1, info["num_ctas"], flags)
    for _ in range(2):
        o, l, i = _static(cfg, tables, q, kv)
        assert i["num_items"] == info["num_items"]
        _close(o, l, ref_o, ref_l)
        _against_oracle(w, tables, q, kv, o, l)
    assert _last_error(cfg) == 0


def test_static_scratch_warm_call_allocates_nothing():
    w = _llama_like_small()
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    cfg = pkd.make_config(w.hq, w.hkv, w.head_dim, w.page_size, w.batch,
                          int(t["indptr"][-1]), w.pool_pages, -1, -1, 152)
    words, _, _ = pkd.plan_host(cfg, t["indptr"], t["indices"], t["last"])
    out = torch.empty_like(q)
    lse = torch.empty(w.batch, w.hq, dtype=torch.float32, device="cuda")
    assert _call(cfg, words, q, kv, out, lse) == 0      # first call: set-up, kernels loaded
    torch.cuda.synchronize()
    torch_before = torch.cuda.memory_allocated()
    free_before = torch.cuda.mem_get_info()[0]
    assert _call(cfg, words, q, kv, out, lse) == 0
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == torch_before
    assert torch.cuda.mem_get_info()[0] == free_before


def test_static_scratch_reports_device_errors():
    """A schedule whose page ids lie past the pool the run is given: the
    decode kernel's range check skips those pages and flags them, and the
    error reader returns (then clears) the flag."""
    w = _llama_like_small()
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    nnz = int(t["indptr"][-1])
    cfg = pkd.make_config(w.hq, w.hkv, w.head_dim, w.page_size, w.batch, nnz, w.pool_pages,
                          -1, -1, 152)
    big = pkd.make_config(w.hq, w.hkv, w.head_dim, w.page_size, w.batch, nnz,
                          w.pool_pages + 64, -1, -1, 152)
    bad_indices = np.array(t["indices"], np.int32).copy()
    bad_indices[0] = w.pool_pages + 5             # outside the run's pool
    words, _, _ = pkd.plan_host(big, t["indptr"], bad_indices, t["last"])
    out = torch.empty_like(q)
    lse = torch.empty(w.batch, w.hq, dtype=torch.float32, device="cuda")
    assert _call(cfg, words, q, kv, out, lse) == 0
    assert _last_error(cfg) == pkd.DEV_ERR_BOUNDS
    assert _last_error(cfg) == 0                  # read clears it


def test_static_scratch_rejects_oversized_layout():
    lib = pkd.load()
    # 512 requests x 64 query heads of partial states: far above 32 MiB
    cfg = pkd.make_config(64, 8, 128, 1, 4096, 1 << 20, 1 << 20, -1, -1, 152)
    words = np.zeros(16, dtype=np.int32)
    q = torch.empty(1, 64, 128, dtype=torch.bfloat16, device="cuda")
    st = lib.pkd_run_static_scratch(ctypes.byref(cfg), ctypes.c_void_p(words.ctypes.data),
                                    words.size, ctypes.c_void_p(q.data_ptr()),
                                    ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(q.data_ptr()),
                                    None, None)
    assert st == -10                                   # PKD_E_SCRATCH_LIMIT
