"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Tolerances (stated for this path): max-abs error <= 2e-2 on the bf16
outputs, <= 1e-3 on the fp32 LSE.  Every test compares every output element:
the small cases, and the full-size workloads in the launch configuration the
benchmark uses (default CTA count, CUDA graph for the 32-layer step, whose
first and last layers are checked in full).
"""
import math

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


def _decoder(w, indptr, *, num_ctas=0, alpha=-1, min_chunk=-1, max_batch=None, max_pages=None,
             tc=None):
    return pkd.BatchDecodeWithPagedKVCache(
        w.hq, w.hkv, w.head_dim, w.page_size,
        max_batch=max_batch or max(w.batch, 1),
        max_num_pages=max_pages or max(int(indptr[-1]), 1),
        num_pages=w.pool_pages, num_ctas=num_ctas, alpha=alpha, min_chunk_tokens=min_chunk,
        use_tensor_cores=tc)


def _check(out, lse, ref_o, ref_l, rows=None):
    o = out.double().cpu().numpy()
    l = lse.double().cpu().numpy()
    if rows is not None:
        o = o[rows[:, 0], rows[:, 1]]
        l = l[rows[:, 0], rows[:, 1]]
    assert np.isfinite(o).all() and np.isfinite(l).all()
    eo = np.abs(o - ref_o).max() if o.size else 0.0
    el = np.abs(l - ref_l).max() if l.size else 0.0
    assert eo <= OUT_TOL, f"out max-abs {eo}"
    assert el <= LSE_TOL, f"lse max-abs {el}"
    return eo, el


def _small_case(seed, lens, P, hq, hkv, scale_q=1.0):
    w = workloads.Workload(f"s{seed}", seed, hq, hkv, 128, P, 1, tuple(lens),
                           sum(-(-l // P) for l in lens) + 5)
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    if scale_q != 1.0:
        q = (q.float() * scale_q).to(torch.bfloat16)
    kv = workloads.make_kv(w, device="cuda")[0]
    return w, t, q, kv


SMALL = [
    # (seed, lens, P, Hq, Hkv)
    (1, [37, 16, 5], 16, 32, 8),                  # worked example shape
    (2, [1, 2, 15, 16, 17, 31, 33, 100], 16, 32, 8),
    (3, [300, 7, 1024, 5], 1, 64, 8),              # token-level sparse, g = 8
    (4, [513, 97, 2000], 3, 8, 8),                 # odd page size, g = 1
    (5, [700, 41, 1], 32, 16, 8),                  # pages longer than a stage
    (6, [900, 260, 35], 16, 16, 4),                # 4 KV heads, g = 4
    (7, [450, 18], 8, 4, 2),                       # 2 KV heads, g = 2
    (8, [333, 5, 64], 16, 8, 1),                   # MQA, g = 8
]


@pytest.mark.parametrize("case", SMALL, ids=[f"case{c[0]}" for c in SMALL])
@pytest.mark.parametrize("split", ["writethrough", "split"])
@pytest.mark.parametrize("tc", [False, True], ids=["fma", "mma"])
def test_small_parity_every_element(case, split, tc):
    """Every element, both consumer variants (CUDA-core FMA and tensor-core
    MMA folding of the GQA group), with and without split-KV."""
    seed, lens, P, hq, hkv = case
    w, t, q, kv = _small_case(seed, lens, P, hq, hkv)
    kw = dict(num_ctas=1, min_chunk=1 << 30) if split == "writethrough" else \
        dict(num_ctas=5, alpha=0, min_chunk=1)
    dec = _decoder(w, t["indptr"], tc=tc, **kw)
    dec.plan(t["indptr"], t["indices"], t["last"])
    info = dec.plan_info()
    if split == "split" and max(lens) > 64:
        assert info["num_units"] >= 1
    out, lse = dec.run(q, kv)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=hq, hkv=hkv)
    _check(out, lse, ref_o, ref_l)
    assert dec.device_error() == 0


@pytest.mark.parametrize("tc", [False, True], ids=["fma", "mma"])
def test_peaky_scores_parity(tc):
    w, t, q, kv = _small_case(11, [640, 77, 1500], 16, 32, 8, scale_q=8.0)
    dec = _decoder(w, t["indptr"], num_ctas=6, alpha=0, min_chunk=1, tc=tc)
    dec.plan(t["indptr"], t["indices"], t["last"])
    out, lse = dec.run(q, kv)
    ref_o, ref_l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=32, hkv=8)
    _check(out, lse, ref_o, ref_l)


def test_split_equals_unsplit_and_determinism():
    w, t, q, kv = _small_case(12, [4000, 123, 2500, 16], 16, 32, 8)
    a = _decoder(w, t["indptr"], num_ctas=1, min_chunk=1 << 30)
    b = _decoder(w, t["indptr"], num_ctas=16, alpha=0, min_chunk=16)
    a.plan(t["indptr"], t["indices"], t["last"])
    b.plan(t["indptr"], t["indices"], t["last"])
    assert a.plan_info()["num_units"] == 0 and b.plan_info()["num_units"] >= 2
    oa, la = a.run(q, kv)
    ob, lb = b.run(q, kv)
    ob2, lb2 = b.run(q, kv)
    torch.cuda.synchronize()
    # run twice -> bit-identical (fixed reduction map, no atomics)
    assert torch.equal(ob, ob2) and torch.equal(lb, lb2)
    assert (oa.float() - ob.float()).abs().max().item() <= OUT_TOL
    assert (la - lb).abs().max().item() <= LSE_TOL
    ref_o, ref_l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=32, hkv=8)
    _check(oa, la, ref_o, ref_l)
    _check(ob, lb, ref_o, ref_l)


def test_device_schedule_matches_host_planner():
    w = workloads.workload("skewed")
    t = workloads.make_tables(w)
    dec = _decoder(w, t["indptr"])
    dec.plan(t["indptr"], t["indices"], t["last"])
    words, info, off = dec.schedule()
    cfg = pkd.make_config(w.hq, w.hkv, 128, w.page_size, w.batch, int(t["indptr"][-1]),
                          w.pool_pages, -1, -1, info["num_ctas"])
    hwords, hinfo, hoff = pkd.plan_host(cfg, t["indptr"], t["indices"], t["last"])
    assert off == hoff
    n = off[4] + info["nnz"]
    assert words[21] == 1                     # the device header carries the plan's epoch
    hwords[21] = words[21]                    # (host-only plans leave it 0)
    np.testing.assert_array_equal(words[:n], hwords[:n])
    from oracle import plan as oplan
    ref = oplan.plan(t["indptr"], t["indices"], t["last"], page_size=16,
                     num_pages=w.pool_pages, n_cta=info["num_ctas"], alpha=32,
                     min_chunk_tokens=256)
    assert pkd.decode_schedule(words, off, info)["page_list"] == ref.page_list


def test_empty_batch():
    w, t, q, kv = _small_case(13, [20], 16, 32, 8)
    dec = _decoder(w, t["indptr"])
    empty = np.zeros(1, np.int32)
    dec.plan(empty, np.zeros(0, np.int32), np.zeros(0, np.int32))
    q0 = torch.empty(0, 32, 128, dtype=torch.bfloat16, device="cuda")
    out, lse = dec.run(q0, kv)
    torch.cuda.synchronize()
    assert out.shape == (0, 32, 128)
    assert dec.device_error() == 0


# ------------------------------------------------------------- full sizes

@pytest.mark.parametrize("tc", [None, False], ids=["default", "fma"])
def test_skewed_full_parity(tc):
    """63 short requests + one 100,000-token request, default grid."""
    w = workloads.workload("skewed")
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    dec = _decoder(w, t["indptr"], tc=tc)
    dec.plan(t["indptr"], t["indices"], t["last"])
    assert dec.plan_info()["num_units"] >= 1
    out, lse = dec.run(q, kv)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=32, hkv=8)
    _check(out, lse, ref_o, ref_l)
    assert dec.device_error() == 0


def test_llama8b_step_graph_full_parity():
    """32-layer step under CUDA-graph replay, as the benchmark runs it: every
    output of the first and the last layer (64 requests x 32 query heads each)
    against the oracle."""
    w = workloads.workload("llama8b_step")
    t = workloads.make_tables(w)
    qs = workloads.make_q(w, device="cuda")
    kvs = workloads.make_kv(w, device="cuda")
    outs = [torch.empty_like(x) for x in qs]
    lses = [torch.empty(w.batch, w.hq, dtype=torch.float32, device="cuda") for _ in qs]
    dec = _decoder(w, t["indptr"])
    dec.plan(t["indptr"], t["indices"], t["last"])
    g = dec.capture(qs, kvs, outs, lses, timing=True)
    dec.plan(t["indptr"], t["indices"], t["last"])   # re-plan in place, then replay
    g.launch()
    torch.cuda.synchronize()
    assert all(x > 0 for x in g.layer_times())
    assert dec.plan_info()["num_units"] >= 1       # split requests go through the merge
    for layer in (0, 31):
        ref_o, ref_l = oracle.decode(qs[layer], kvs[layer], t["indptr"], t["indices"],
                                     t["last"], hq=32, hkv=8)
        _check(outs[layer], lses[layer], ref_o, ref_l)
    # the graph gives the same bits as direct runs
    o_direct, l_direct = dec.run(qs[5], kvs[5])
    torch.cuda.synchronize()
    assert torch.equal(o_direct, outs[5]) and torch.equal(l_direct, lses[5])
    g.close()
    assert dec.device_error() == 0


def test_shared_prefix_merge_states_parity():
    """Prefix view and suffix view run separately, combined by merge_states."""
    w = workloads.workload("shared_prefix")
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    pre = _decoder(w, t["prefix"][0])
    suf = _decoder(w, t["suffix"][0])
    pre.plan(*t["prefix"])
    suf.plan(*t["suffix"])
    op, lp = pre.run(q, kv)
    os_, ls = suf.run(q, kv)
    out, lse = pkd.merge_states(op, lp, os_, ls)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=32, hkv=8)
    _check(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("tc", [None, False], ids=["default", "fma"])
def test_token_sparse_full_parity(tc):
    """Page size 1, 512 requests, g = 8: every output (512 x 64 rows)."""
    w = workloads.workload("token_sparse")
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    dec = _decoder(w, t["indptr"], tc=tc)
    dec.plan(t["indptr"], t["indices"], t["last"])
    out, lse = dec.run(q, kv)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=64, hkv=8)
    _check(out, lse, ref_o, ref_l)
    assert dec.device_error() == 0


# ------------------------------------------------------------- merge_states

def test_merge_states_against_oracle():
    g = torch.Generator(device="cuda").manual_seed(9)
    n, H, D = 33, 12, 128
    va = torch.randn(n, H, D, generator=g, device="cuda").to(torch.bfloat16)
    vb = torch.randn(n, H, D, generator=g, device="cuda").to(torch.bfloat16)
    sa = torch.randn(n, H, generator=g, device="cuda") * 4
    sb = torch.randn(n, H, generator=g, device="cuda") * 4
    sa[0, :3] = -math.inf                  # empty left state
    sb[1, :2] = -math.inf                  # empty right state
    sa[2, 0] = -math.inf
    sb[2, 0] = -math.inf                   # both empty
    vo, so = pkd.merge_states(va, sa, vb, sb)
    torch.cuda.synchronize()
    ro, rl = oracle.merge(va.double().cpu().numpy(), sa.double().cpu().numpy(),
                          vb.double().cpu().numpy(), sb.double().cpu().numpy())
    o = vo.double().cpu().numpy()
    l = so.double().cpu().numpy()
    fin = np.isfinite(rl)
    assert np.abs(o - ro).max() <= OUT_TOL
    assert np.abs(l[fin] - rl[fin]).max() <= LSE_TOL
    assert np.all(np.isneginf(l[~fin])) and np.all(o[~fin] == 0)
    # in place (outputs alias the first state)
    va2, sa2 = va.clone(), sa.clone()
    pkd.merge_states(va2, sa2, vb, sb, v_out=va2, s_out=sa2)
    torch.cuda.synchronize()
    assert torch.equal(va2, vo) and torch.equal(sa2, so)


def test_merge_paths_at_the_32_chunk_boundary():
    """A request split into 32 chunks is folded by one warp, one split into
    33 by a whole block: both against the oracle."""
    lens = [512, 528, 40]
    w = workloads.Workload("m32", 77, 32, 8, 128, 16, 1, tuple(lens),
                           sum(-(-l // 16) for l in lens) + 2)
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    dec = pkd.BatchDecodeWithPagedKVCache(w.hq, w.hkv, 128, 16, max_batch=3,
                                          max_num_pages=int(t["indptr"][-1]),
                                          num_pages=w.pool_pages, num_ctas=68, alpha=0,
                                          min_chunk_tokens=16, chunk_rule="search")
    dec.plan(t["indptr"], t["indices"], t["last"])
    info = dec.plan_info()
    assert info["chunk_tokens"] == 16
    words, info, off = dec.schedule()
    units = pkd.decode_schedule(words, off, info)["units"]
    assert sorted(n for _, n in units) == [3, 32, 33]
    out, lse = dec.run(q, kv)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=32, hkv=8)
    _check(out, lse, ref_o, ref_l)


def test_merge_batched_loads_for_long_units():
    """A plan with a request split into more than 64 chunks takes the merge
    whose warps keep several slots' loads in flight (units of 64, 65 and 130
    chunks in one plan), against the oracle."""
    lens = [1024, 1040, 2080, 40]
    w = workloads.Workload("m130", 79, 32, 8, 128, 16, 1, tuple(lens),
                           sum(-(-l // 16) for l in lens) + 2)
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    dec = pkd.BatchDecodeWithPagedKVCache(w.hq, w.hkv, 128, 16, max_batch=4,
                                          max_num_pages=int(t["indptr"][-1]),
                                          num_pages=w.pool_pages, num_ctas=152, alpha=0,
                                          min_chunk_tokens=16, chunk_rule="search")
    dec.plan(t["indptr"], t["indices"], t["last"])
    words, info, off = dec.schedule()
    assert info["chunk_tokens"] == 16
    units = pkd.decode_schedule(words, off, info)["units"]
    assert sorted(n for _, n in units) == [3, 64, 65, 130]
    out, lse = dec.run(q, kv)
    out2, lse2 = dec.run(q, kv)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    ref_o, ref_l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=32, hkv=8)
    _check(out, lse, ref_o, ref_l)


def test_merge_warp_mode_many_units():
    """At least 4 merge tasks per merge block: the warp-per-task merge,
    against the oracle on every element (20 requests, 16 split, Hq 16 ->
    256 tasks for 8 CTAs x 8 merge blocks)."""
    rng = np.random.default_rng(20)
    lens = rng.integers(200, 1200, 20).tolist()
    w = workloads.Workload("mw", 78, 16, 2, 128, 16, 1, tuple(lens),
                           sum(-(-l // 16) for l in lens) + 2)
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    dec = pkd.BatchDecodeWithPagedKVCache(w.hq, w.hkv, 128, 16, max_batch=w.batch,
                                          max_num_pages=int(t["indptr"][-1]),
                                          num_pages=w.pool_pages, num_ctas=8, alpha=0,
                                          min_chunk_tokens=16)
    dec.plan(t["indptr"], t["indices"], t["last"])
    info = dec.plan_info()
    assert info["num_units"] * w.hq >= 4 * 8 * 8      # tasks >= 4 x merge blocks
    out, lse = dec.run(q, kv)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=w.hq, hkv=w.hkv)
    _check(out, lse, ref_o, ref_l)
