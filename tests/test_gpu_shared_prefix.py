"""GPU parity of the shared-prefix (composable-format) path.

A shared-prefix context plans groups of requests over one page list per
group; its run returns each request's attention state over the group's
pages, which merge_states combines with the request's own suffix state.
Checked against the fp64 oracle (2e-2 on bf16 out, 1e-3 on fp32 lse)."""
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


def _check(out, lse, ref_o, ref_l):
    o = out.double().cpu().numpy()
    l = lse.double().cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(l).all()
    assert np.abs(o - ref_o).max() <= OUT_TOL, np.abs(o - ref_o).max()
    assert np.abs(l - ref_l).max() <= LSE_TOL, np.abs(l - ref_l).max()


def _expand(group_indptr, indptr, indices, last):
    """Per-request table: request r of group j owns group j's pages."""
    rows_ip, rows_ix, rows_last = [0], [], []
    for j in range(len(last)):
        for _ in range(group_indptr[j], group_indptr[j + 1]):
            rows_ix.extend(indices[indptr[j]:indptr[j + 1]].tolist())
            rows_ip.append(len(rows_ix))
            rows_last.append(int(last[j]))
    return (np.array(rows_ip, np.int32), np.array(rows_ix, np.int32),
            np.array(rows_last, np.int32))


CASES = [
    # (seed, group sizes, group lengths, P, Hq, Hkv, n_cta)
    (1, [32], [8192], 16, 32, 8, 0),             # the workload's shape, default grid
    (2, [5, 3, 9], [700, 33, 2048], 16, 32, 8, 7),
    (3, [6, 2], [900, 1500], 1, 64, 8, 9),        # g = 8, token-level pages
    (4, [17, 4], [1200, 64], 16, 16, 8, 5),       # g = 2
    (5, [20], [333], 3, 8, 8, 3),                 # g = 1
    (6, [3, 11], [4000, 100], 16, 16, 4, 6),      # 4 KV heads
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{c[0]}" for c in CASES])
def test_prefix_states_match_oracle(case):
    seed, sizes, glens, P, hq, hkv, n_cta = case
    rng = np.random.default_rng(seed)
    B = sum(sizes)
    group_indptr = np.array([0] + np.cumsum(sizes).tolist(), np.int32)
    pool = sum(-(-l // P) for l in glens) + 3
    indptr, indices, last = workloads.page_table(glens, P, rng.permutation(pool).astype(np.int32))
    w = workloads.Workload(f"sp{seed}", 60 + seed, hq, hkv, 128, P, 1, tuple([1] * B), pool)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    dec = pkd.BatchDecodeWithPagedKVCache(hq, hkv, 128, P, max_batch=B,
                                          max_num_pages=int(indptr[-1]), num_pages=pool,
                                          num_ctas=n_cta, shared_prefix=True)
    dec.plan_shared(group_indptr, indptr, indices, last)
    out, lse = dec.run(q, kv)
    out2, lse2 = dec.run(q, kv)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)      # deterministic
    e_ip, e_ix, e_last = _expand(group_indptr, indptr, indices, last)
    ref_o, ref_l = oracle.decode(q, kv, e_ip, e_ix, e_last, hq=hq, hkv=hkv)
    _check(out, lse, ref_o, ref_l)
    assert dec.device_error() == 0


def test_shared_prefix_workload_composed():
    """Prefix level (one group of 32 requests over 512 shared pages) through
    the shared-prefix kernel, suffixes through the decode kernel,
    merge_states: equals attention over prefix + suffix."""
    w = workloads.workload("shared_prefix")
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    P = w.page_size
    n_pre = w.prefix_tokens // P
    pre_pages = t["prefix"][1][:n_pre]
    g_ip = np.array([0, w.batch], np.int32)
    p_ip = np.array([0, n_pre], np.int32)
    p_last = np.array([P], np.int32)
    pre = pkd.BatchDecodeWithPagedKVCache(w.hq, w.hkv, 128, P, max_batch=w.batch,
                                          max_num_pages=n_pre, num_pages=w.pool_pages,
                                          shared_prefix=True)
    suf = pkd.BatchDecodeWithPagedKVCache(w.hq, w.hkv, 128, P, max_batch=w.batch,
                                          max_num_pages=int(t["suffix"][0][-1]),
                                          num_pages=w.pool_pages)
    pre.plan_shared(g_ip, p_ip, pre_pages, p_last)
    suf.plan(*t["suffix"])
    op, lp = pre.run(q, kv)
    os_, ls = suf.run(q, kv)
    out, lse = pkd.merge_states(op, lp, os_, ls)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=w.hq, hkv=w.hkv)
    _check(out, lse, ref_o, ref_l)


def test_plan_shared_needs_shared_context_and_valid_groups():
    dec = pkd.BatchDecodeWithPagedKVCache(32, 8, 128, 16, max_batch=8, max_num_pages=8,
                                          num_pages=8)
    with pytest.raises(pkd.PkdError):
        dec.plan_shared(np.array([0, 2], np.int32), np.array([0, 1], np.int32),
                        np.array([0], np.int32), np.array([4], np.int32))
    sp = pkd.BatchDecodeWithPagedKVCache(32, 8, 128, 16, max_batch=8, max_num_pages=8,
                                         num_pages=8, shared_prefix=True)
    for gi in ([0, 0], [1, 3], [0, 9]):       # empty group, bad start, above capacity
        with pytest.raises(pkd.PkdError):
            sp.plan_shared(np.array(gi, np.int32), np.array([0, 1], np.int32),
                           np.array([0], np.int32), np.array([4], np.int32))
    with pytest.raises(pkd.PkdError):          # FMA consumer has no shared-prefix kernel
        pkd.BatchDecodeWithPagedKVCache(32, 8, 128, 16, max_batch=8, max_num_pages=8,
                                        num_pages=8, shared_prefix=True, use_tensor_cores=False)
