"""GPU parity of the dense shared-prefix kernel (tcgen05 tensor cores,
tensor-memory accumulators; PKD_FLAG_DENSE_PREFIX) against the fp64 oracle:
groups of requests over shared page tables, every request's state over its
group's tokens.  Tolerances as everywhere: 2e-2 on bf16 out, 1e-3 on lse."""
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


def _expand(sizes, indptr, indices, last):
    e_ip, e_ix, e_last = [0], [], []
    for j in range(len(sizes)):
        for _ in range(sizes[j]):
            e_ix.extend(indices[indptr[j]:indptr[j + 1]].tolist())
            e_ip.append(len(e_ix))
            e_last.append(int(last[j]))
    return (np.array(e_ip, np.int32), np.array(e_ix, np.int32), np.array(e_last, np.int32))


def _poison_tails(kv, indptr, indices, last, P, hnd):
    for j in range(len(last)):
        page = int(indices[int(indptr[j + 1]) - 1])
        if int(last[j]) < P:
            if hnd:
                kv[page, :, :, int(last[j]):] = float("nan")
            else:
                kv[page, :, int(last[j]):] = float("nan")


CASES = [
    # (seed, group sizes, group lengths, P, Hq, Hkv, n_cta, layout)
    (1, [32], [8192], 16, 32, 8, 0, "NHD"),          # the workload's shape, default grid
    (2, [5, 3, 9], [700, 33, 2047], 16, 32, 8, 7, "NHD"),
    (3, [40, 2], [1500, 64], 16, 16, 8, 9, "NHD"),    # g = 2: blocks of 64 requests
    (4, [150, 7], [333, 1200], 32, 8, 8, 5, "NHD"),   # g = 1: blocks of 128, two blocks
    (5, [20], [999], 16, 64, 8, 3, "NHD"),            # g = 8: blocks of 16
    (6, [3, 11], [4000, 100], 64, 16, 4, 6, "HND"),   # 4 KV heads, HND, 4 tiles per page
    (7, [1, 1, 1], [17, 1, 16], 16, 32, 8, 4, "NHD"),  # tiny: one partial tile each
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{c[0]}" for c in CASES])
def test_dense_prefix_states_match_oracle(case):
    seed, sizes, glens, P, hq, hkv, n_cta, layout = case
    rng = np.random.default_rng(seed)
    B = sum(sizes)
    group_indptr = np.array([0] + np.cumsum(sizes).tolist(), np.int32)
    pool = sum(-(-l // P) for l in glens) + 3
    indptr, indices, last = workloads.page_table(glens, P, rng.permutation(pool).astype(np.int32))
    w = workloads.Workload(f"dp{seed}", 800 + seed, hq, hkv, 128, P, 1, tuple([1] * B), pool,
                           kv_layout=layout)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    e_ip, e_ix, e_last = _expand(sizes, indptr, indices, last)
    ref_o, ref_l = oracle.decode(q, kv, e_ip, e_ix, e_last, hq=hq, hkv=hkv, layout=layout)
    _poison_tails(kv, indptr, indices, last, P, layout == "HND")
    dec = pkd.BatchDecodeWithPagedKVCache(hq, hkv, 128, P, max_batch=B,
                                          max_num_pages=int(indptr[-1]), num_pages=pool,
                                          num_ctas=n_cta, shared_prefix=True, dense_prefix=True,
                                          kv_layout=layout)
    dec.plan_shared(group_indptr, indptr, indices, last)
    out, lse = dec.run(q, kv)
    out2, lse2 = dec.run(q, kv)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)      # deterministic
    _check(out, lse, ref_o, ref_l)
    assert dec.device_error() == 0


def test_dense_prefix_search_rule_and_scaled_values():
    """Binary-search chunks and peaky scores (q x 8: the running max grows,
    so the rescale path runs)."""
    sizes, glens, P, hq, hkv = [12, 30], [5000, 2500], 16, 32, 8
    rng = np.random.default_rng(31)
    B = sum(sizes)
    group_indptr = np.array([0] + np.cumsum(sizes).tolist(), np.int32)
    pool = sum(-(-l // P) for l in glens) + 3
    indptr, indices, last = workloads.page_table(glens, P, rng.permutation(pool).astype(np.int32))
    w = workloads.Workload("dps", 840, hq, hkv, 128, P, 1, tuple([1] * B), pool)
    q = (workloads.make_q(w, device="cuda")[0].float() * 8.0).to(torch.bfloat16)
    kv = workloads.make_kv(w, device="cuda")[0]
    dec = pkd.BatchDecodeWithPagedKVCache(hq, hkv, 128, P, max_batch=B,
                                          max_num_pages=int(indptr[-1]), num_pages=pool,
                                          shared_prefix=True, dense_prefix=True,
                                          chunk_rule="search")
    dec.plan_shared(group_indptr, indptr, indices, last)
    assert dec.plan_info()["num_units"] >= 1
    out, lse = dec.run(q, kv)
    e_ip, e_ix, e_last = _expand(sizes, indptr, indices, last)
    ref_o, ref_l = oracle.decode(q, kv, e_ip, e_ix, e_last, hq=hq, hkv=hkv)
    _check(out, lse, ref_o, ref_l)


def test_dense_prefix_workload_composed_and_graph():
    """The shared-prefix workload: the prefix level on the dense kernel
    (captured in a graph), the suffixes on the decode kernel, merge_states."""
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
                                          shared_prefix=True, dense_prefix=True)
    suf = pkd.BatchDecodeWithPagedKVCache(w.hq, w.hkv, 128, P, max_batch=w.batch,
                                          max_num_pages=int(t["suffix"][0][-1]),
                                          num_pages=w.pool_pages)
    pre.plan_shared(g_ip, p_ip, pre_pages, p_last)
    suf.plan(*t["suffix"])
    op = torch.empty_like(q)
    lp = torch.empty(w.batch, w.hq, dtype=torch.float32, device="cuda")
    g = pre.capture([q], [kv], [op], [lp])
    g.launch()
    os_, ls = suf.run(q, kv)
    out, lse = pkd.merge_states(op, lp, os_, ls)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=w.hq, hkv=w.hkv)
    _check(out, lse, ref_o, ref_l)
    # a plan with another batch makes the captured query maps stale
    pre.plan_shared(np.array([0, w.batch - 1], np.int32), p_ip, pre_pages, p_last)
    with pytest.raises(pkd.PkdError) as e:
        g.launch()
    assert e.value.status == -6
    g.close()
    assert pre.device_error() == 0


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_dense_prefix_longest_sweep_case(layout):
    """The largest case of the composable-format sweep: 64 requests over a
    32,768-token prefix (two 128-row tiles per KV head, items of ~20
    128-token rounds, every ring slot reused many times), each with its own
    128-token suffix; prefix level on the dense kernel, suffixes on the
    decode kernel, merge_states; every output against the oracle."""
    w = workloads.shared_prefix_case(32768, 64)
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    P = w.page_size
    n_pre = w.prefix_tokens // P
    hnd = layout == "HND"
    if hnd:   # the same values in the HND layout: [pages, 2, Hkv, P, D]
        kv = kv.permute(0, 1, 3, 2, 4).contiguous()
    pre = pkd.BatchDecodeWithPagedKVCache(w.hq, w.hkv, 128, P, max_batch=w.batch,
                                          max_num_pages=n_pre, num_pages=w.pool_pages,
                                          shared_prefix=True, dense_prefix=True,
                                          kv_layout=layout)
    suf = pkd.BatchDecodeWithPagedKVCache(w.hq, w.hkv, 128, P, max_batch=w.batch,
                                          max_num_pages=int(t["suffix"][0][-1]),
                                          num_pages=w.pool_pages, kv_layout=layout)
    pre.plan_shared(np.array([0, w.batch], np.int32), np.array([0, n_pre], np.int32),
                    t["prefix"][1][:n_pre], np.array([P], np.int32))
    info = pre.plan_info()
    assert info["num_units"] == w.batch            # every request's prefix is split
    suf.plan(*t["suffix"])
    op, lp = pre.run(q, kv)
    os_, ls = suf.run(q, kv)
    out, lse = pkd.merge_states(op, lp, os_, ls)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=w.hq, hkv=w.hkv,
                                 layout=layout)
    _check(out, lse, ref_o, ref_l)
    assert pre.device_error() == 0 and suf.device_error() == 0


def test_dense_prefix_rejects_unsupported():
    with pytest.raises(ValueError):
        pkd.BatchDecodeWithPagedKVCache(32, 8, 128, 16, max_batch=4, max_num_pages=8,
                                        num_pages=8, dense_prefix=True)
    with pytest.raises(pkd.PkdError):            # page tiles need P % 16 == 0
        pkd.BatchDecodeWithPagedKVCache(32, 8, 128, 8, max_batch=4, max_num_pages=8,
                                        num_pages=8, shared_prefix=True, dense_prefix=True)
    with pytest.raises(pkd.PkdError):            # bf16 cache only
        pkd.BatchDecodeWithPagedKVCache(32, 8, 128, 16, max_batch=4, max_num_pages=8,
                                        num_pages=8, shared_prefix=True, dense_prefix=True,
                                        kv_dtype="e4m3")


def test_dense_prefix_run_waits_on_the_device_for_a_plan_from_another_stream():
    """The standalone dense kernel with a plan uploaded on a side stream held
    back by a GPU sleep and the run issued on another stream with
    expect_epoch and no event: it computes the new plan (two groups) rather
    than the one already in the workspace (one group of all requests)."""
    sizes, glens, P, hq, hkv = [12, 30], [5000, 2500], 16, 32, 8
    rng = np.random.default_rng(41)
    B = sum(sizes)
    pool = sum(-(-l // P) for l in glens) + 3
    indptr, indices, last = workloads.page_table(glens, P, rng.permutation(pool).astype(np.int32))
    w = workloads.Workload("dpx", 841, hq, hkv, 128, P, 1, tuple([1] * B), pool)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    dec = pkd.BatchDecodeWithPagedKVCache(hq, hkv, 128, P, max_batch=B,
                                          max_num_pages=int(indptr[-1]), num_pages=pool,
                                          shared_prefix=True, dense_prefix=True)
    # first plan: every request over group 0's pages
    dec.plan_shared(np.array([0, B], np.int32), indptr[:2], indices, last[:1])
    dec.run(q, kv)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((B, hq), float("nan"), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    side, main = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(side):
        torch.cuda._sleep(int(1e8))
    ep = dec.plan_shared(np.array([0] + np.cumsum(sizes).tolist(), np.int32), indptr, indices,
                         last, stream=side)
    dec.run(q, kv, out=out, lse=lse, expect_epoch=ep, stream=main)
    held_back = not side.query()
    torch.cuda.synchronize()
    assert held_back, "the upload had already landed when the run was issued"
    e_ip, e_ix, e_last = _expand(sizes, indptr, indices, last)
    ref_o, ref_l = oracle.decode(q, kv, e_ip, e_ix, e_last, hq=hq, hkv=hkv)
    _check(out, lse, ref_o, ref_l)
    assert dec.device_error() == 0
