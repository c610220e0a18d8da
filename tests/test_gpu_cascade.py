"""GPU parity of cascade plans: a shared-prefix level and every request's own
suffix in one schedule, one launch (dense tensor-core role on the first CTAs,
decode role on the others) and one merge, against the fp64 oracle -- every
output element, max-abs 2e-2 on bf16 out and 1e-3 on fp32 lse.

Reference: with the prefix in whole pages, one oracle decode over each
request's full table (prefix pages, then its own).  With a partial last
prefix page (not a paged table any more), the oracle's prefix state and
suffix state of each request, merged by the oracle's merge."""
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
    eo, el = np.abs(o - ref_o).max(), np.abs(l - ref_l).max()
    assert eo <= OUT_TOL, f"out max-abs {eo}"
    assert el <= LSE_TOL, f"lse max-abs {el}"


def _hnd(kv):
    return kv.permute(0, 1, 3, 2, 4).contiguous()


def _workload_tables(w, t):
    n_pre = w.prefix_tokens // w.page_size
    prefix = (np.array([0, n_pre], np.int32), np.asarray(t["prefix"][1][:n_pre], np.int32),
              np.array([w.page_size], np.int32))
    return np.array([0, w.batch], np.int32), prefix, t["suffix"]


def _context(w, gi, prefix, suffix, layout="NHD", num_ctas=0):
    nnz = int(prefix[0][-1]) + int(suffix[0][-1])
    return pkd.BatchDecodeWithPagedKVCache(w.hq, w.hkv, w.head_dim, w.page_size,
                                           max_batch=int(gi[-1]), max_num_pages=nnz,
                                           num_pages=w.pool_pages, cascade=True,
                                           kv_layout=layout, num_ctas=num_ctas)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_cascade_shared_prefix_workload_every_element(layout):
    """32 requests over an 8,192-token shared prefix plus their suffixes:
    against one oracle decode over each request's full table."""
    w = workloads.workload("shared_prefix")
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    gi, prefix, suffix = _workload_tables(w, t)
    dec = _context(w, gi, prefix, suffix, layout)
    dec.plan_cascade(gi, prefix, suffix)
    info = dec.plan_info()
    assert 1 <= info["prefix_ctas"] < info["num_ctas"]
    out, lse = dec.run(q, kv if layout == "NHD" else _hnd(kv))
    out2, lse2 = dec.run(q, kv if layout == "NHD" else _hnd(kv))
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)      # fixed reduction map
    ref_o, ref_l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=w.hq,
                                 hkv=w.hkv)
    _check(out, lse, ref_o, ref_l)
    assert dec.device_error() == 0


def _expanded(gi, prefix):
    """The prefix table with one row per request (its group's row)."""
    ip, ix, last = prefix
    e_ip, e_ix, e_last = [0], [], []
    for j in range(len(gi) - 1):
        for _ in range(gi[j], gi[j + 1]):
            e_ix.extend(ix[ip[j]:ip[j + 1]].tolist())
            e_ip.append(len(e_ix))
            e_last.append(int(last[j]))
    return np.array(e_ip, np.int32), np.array(e_ix, np.int32), np.array(e_last, np.int32)


CASES = [
    # (seed, group sizes, prefix lengths, suffix range, Hq, Hkv, CTAs)
    (1, [5, 40, 3], [1000, 4090, 33], (1, 700), 32, 8, 0),
    (2, [70], [12001], (100, 2000), 64, 8, 0),       # g 8: blocks of 16 requests
    (3, [9, 1], [300, 5000], (1, 40), 16, 8, 11),    # g 2, few CTAs
    (4, [33], [16], (1, 5000), 32, 8, 0),            # a one-page prefix
    (5, [130], [2000], (50, 300), 32, 8, 0),         # two blocks of 32 + ... in one group
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{c[0]}" for c in CASES])
def test_cascade_groups_partial_pages_every_element(case):
    seed, sizes, plens, (lo, hi), hq, hkv, n_cta = case
    rng = np.random.default_rng(900 + seed)
    P = 16
    gi = np.array([0] + np.cumsum(sizes).tolist(), np.int32)
    B = int(gi[-1])
    slens = rng.integers(lo, hi + 1, B).tolist()
    n_pp = sum(-(-l // P) for l in plens)
    n_sp = sum(-(-l // P) for l in slens)
    pool = n_pp + n_sp + 5
    ids = rng.permutation(pool).astype(np.int32)
    prefix = workloads.page_table(plens, P, ids[:n_pp])
    suffix = workloads.page_table(slens, P, ids[n_pp:n_pp + n_sp])
    w = workloads.Workload(f"c{seed}", 500 + seed, hq, hkv, 128, P, 1, tuple(slens), pool)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    dec = _context(w, gi, prefix, suffix, num_ctas=n_cta)
    dec.plan_cascade(gi, prefix, suffix)
    out, lse = dec.run(q, kv)
    torch.cuda.synchronize()
    po, pl = oracle.decode(q, kv, *_expanded(gi, prefix), hq=hq, hkv=hkv)
    so, sl = oracle.decode(q, kv, *suffix, hq=hq, hkv=hkv)
    ref_o, ref_l = oracle.merge(po, pl, so, sl)
    _check(out, lse, ref_o, ref_l)
    assert dec.device_error() == 0


def test_cascade_graph_replay_follows_new_plans():
    """A captured cascade step replayed after re-planning other suffix
    lengths (same batch): the launch reads the new split from the schedule,
    and the replay matches a direct run bit for bit and the oracle."""
    w = workloads.workload("shared_prefix")
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    gi, prefix, suffix = _workload_tables(w, t)
    dec = _context(w, gi, prefix, suffix)
    dec.plan_cascade(gi, prefix, suffix)
    out = torch.empty_like(q)
    lse = torch.empty(w.batch, w.hq, dtype=torch.float32, device="cuda")
    g = dec.capture([q], [kv], [out], [lse])
    # the same requests with their suffixes cut to at most 100 tokens
    s_ip, s_ix, s_last = suffix
    lens = [min(100, 16 * (int(s_ip[r + 1] - s_ip[r]) - 1) + int(s_last[r]))
            for r in range(w.batch)]
    short = workloads.page_table(lens, 16, np.concatenate(
        [s_ix[s_ip[r]:s_ip[r] + -(-lens[r] // 16)] for r in range(w.batch)]).astype(np.int32))
    dec.plan_cascade(gi, prefix, short)
    info = dec.plan_info()
    g.launch()
    torch.cuda.synchronize()
    o_direct, l_direct = dec.run(q, kv)
    torch.cuda.synchronize()
    assert torch.equal(o_direct, out) and torch.equal(l_direct, lse)
    po, pl = oracle.decode(q, kv, *_expanded(gi, prefix), hq=w.hq, hkv=w.hkv)
    so, sl = oracle.decode(q, kv, *short, hq=w.hq, hkv=w.hkv)
    ref_o, ref_l = oracle.merge(po, pl, so, sl)
    _check(out, lse, ref_o, ref_l)
    assert info["prefix_ctas"] >= 1
    g.close()
    assert dec.device_error() == 0


@pytest.mark.parametrize("prefix_tokens,batch", [(1024, 16), (32768, 64)])
def test_cascade_prefix_sweep_cases(prefix_tokens, batch):
    """The composable-format grid's corners (128-token suffixes), against one
    oracle decode over each request's full table."""
    w = workloads.shared_prefix_case(prefix_tokens, batch)
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    gi, prefix, suffix = _workload_tables(w, t)
    dec = _context(w, gi, prefix, suffix)
    dec.plan_cascade(gi, prefix, suffix)
    out, lse = dec.run(q, kv)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=w.hq,
                                 hkv=w.hkv)
    _check(out, lse, ref_o, ref_l)
    assert dec.device_error() == 0


def test_cascade_run_waits_on_the_device_for_a_plan_from_another_stream():
    """A cascade plan uploaded on a side stream held back by a GPU sleep, and
    the run issued on another stream with expect_epoch and no event: the
    cascade kernel waits for the new schedule (its split H_NPRE included)
    and computes the new plan."""
    w = workloads.workload("shared_prefix")
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    gi, prefix, suffix = _workload_tables(w, t)
    dec = _context(w, gi, prefix, suffix)
    # first plan: the suffixes cut to at most 100 tokens
    s_ip, s_ix, s_last = suffix
    lens = [min(100, 16 * (int(s_ip[r + 1] - s_ip[r]) - 1) + int(s_last[r]))
            for r in range(w.batch)]
    short = workloads.page_table(lens, 16, np.concatenate(
        [s_ix[s_ip[r]:s_ip[r] + -(-lens[r] // 16)] for r in range(w.batch)]).astype(np.int32))
    dec.plan_cascade(gi, prefix, short)
    dec.run(q, kv)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.batch, w.hq), float("nan"), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    side, main = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(side):
        torch.cuda._sleep(int(1e8))
    ep = dec.plan_cascade(gi, prefix, suffix, stream=side)      # the full suffixes
    dec.run(q, kv, out=out, lse=lse, expect_epoch=ep, stream=main)
    held_back = not side.query()
    torch.cuda.synchronize()
    assert held_back, "the upload had already landed when the run was issued"
    ref_o, ref_l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=w.hq,
                                 hkv=w.hkv)
    _check(out, lse, ref_o, ref_l)
    assert dec.device_error() == 0
