"""The allocation-free entry point, pkd_run_static_scratch.

It serves callers that may not allocate device memory (an engine whose
allocator owns the whole GPU, a process under a hard memory cap, a plugin
with no allocator): instead of a caller-provided workspace it keeps the
schedule and the split partial states in a static device array inside the
library.  Here it is called through the C ABI twice in a row -- the second
call on a different batch, so stale contents of the shared array from the
first call would show -- and each result is compared with the regular entry
point (pkd_run on a workspace) within the parity tolerances used throughout
the tests (2e-2 on bf16 outputs, 1e-3 on fp32 LSE).

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

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


def _regular(w, tables, q, kv, n_cta):
    ip, ix, la = tables
    dec = pkd.BatchDecodeWithPagedKVCache(w.hq, w.hkv, w.head_dim, w.page_size,
                                          max_batch=w.batch, max_num_pages=int(ip[-1]),
                                          num_pages=w.pool_pages, num_ctas=n_cta)
    dec.plan(ip, ix, la)
    out, lse = dec.run(q, kv)
    torch.cuda.synchronize()
    return out, lse, dec.plan_info()


def _static(cfg, tables, q, kv):
    lib = pkd.load()
    words, info, off = pkd.plan_host(cfg, *tables)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((q.shape[0], q.shape[1]), float("nan"), dtype=torch.float32,
                     device=q.device)
    st = lib.pkd_run_static_scratch(
        ctypes.byref(cfg), ctypes.c_void_p(words.ctypes.data), words.size,
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kv.data_ptr()),
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, pkd.STATUS.get(st, st)
    torch.cuda.synchronize()
    return out, lse, info


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
    assert (o1.float() - ref_o.float()).abs().max().item() <= OUT_TOL
    assert (l1 - ref_l).abs().max().item() <= LSE_TOL

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
    assert (o2.float() - ref_o2.float()).abs().max().item() <= OUT_TOL
    assert (l2 - ref_l2).abs().max().item() <= LSE_TOL


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
