"""Pins for the CPU oracle: it is checked against things other than itself.

* the worked page-table example printed on the pages (golden fixture);
* the length identity l = P (n - 1) + r on the edge lengths the pages call
  out (1, P, P + 1, exact multiples) and the off-by-one failure they warn of;
* brute force: dense attention over K/V gathered page by page into
  contiguous tensors, computed with torch's softmax / logsumexp in fp64;
* closed forms: one token (out = v_0, lse = s_0), identical keys
  (out = mean v, lse = s + ln l);
* the state algebra: merging per-chunk states equals unsplit attention,
  in any order and association; an empty state is the merge identity;
* hand-worked schedules for the plan restatement, plus an exactly-once
  coverage check on random tables.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import plan as oplan

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- page table

def test_worked_example_page_table():
    g = _golden("worked_example.json")
    indptr, indices, last = workloads.page_table(g["kv_lens"], g["page_size"])
    assert indptr.tolist() == g["indptr"]
    assert indices.tolist() == g["indices"]
    assert last.tolist() == g["last_page_len"]
    lens = oracle.lengths(g["indptr"], g["indices"], g["last_page_len"],
                          g["page_size"], num_pages=64)
    assert lens.tolist() == g["kv_lens"]
    assert oplan.lengths(g["indptr"], g["last_page_len"], g["indices"],
                         g["page_size"], 64) == g["kv_lens"]


@pytest.mark.parametrize("P", [1, 4, 16])
def test_length_identity_edges(P):
    lens = [1, max(P - 1, 1), P, P + 1, 2 * P, 3 * P, 100_000]
    indptr, indices, last = workloads.page_table(lens, P)
    assert all(1 <= r <= P for r in last.tolist())
    for i, l in enumerate(lens):
        n = indptr[i + 1] - indptr[i]
        assert n == math.ceil(l / P)
    got = oracle.lengths(indptr, indices, last, P, num_pages=int(indptr[-1]))
    assert got.tolist() == lens
    assert oplan.lengths(indptr, last, indices, P, int(indptr[-1])) == lens


def test_table_errors_rejected():
    P = 16
    # exact multiple of P written with last_page_len = 0 (the off-by-one bug)
    bad_last = ([0, 2], [0, 1], [0])
    good = ([0, 2], [0, 1], [16])
    assert oracle.lengths(*good, P, 4).tolist() == [32]
    with pytest.raises(oracle.OracleError):
        oracle.lengths(*bad_last, P, 4)
    with pytest.raises(oplan.TableError):
        oplan.lengths(bad_last[0], bad_last[2], bad_last[1], P, 4)
    for indptr, indices, last in [
        ([0, 0], [], [1]),            # request owning no page
        ([0, 1], [0], [17]),          # last page longer than the page
        ([0, 1], [4], [1]),           # page id outside the pool
        ([0, 1], [-1], [1]),          # negative page id
        ([1, 2], [0, 1], [1]),        # indptr not starting at 0
    ]:
        with pytest.raises(oracle.OracleError):
            oracle.lengths(indptr, indices, last, P, 4)
        with pytest.raises(oplan.TableError):
            oplan.lengths(indptr, last, indices, P, 4)


# ----------------------------------------------------------- attention pins

def _tiny(seed, lens, P, hq, hkv, D=16, scale_q=1.0):
    w = workloads.Workload(f"t{seed}", seed, hq, hkv, D, P, 1, tuple(lens),
                           sum(math.ceil(l / P) for l in lens) + 2)
    t = workloads.make_tables(w)
    q = workloads.make_q(w)[0]
    if scale_q != 1.0:
        q = (q.float() * scale_q).to(torch.bfloat16)
    kv = workloads.make_kv(w)[0]
    return w, t, q, kv


def _dense_reference(w, t, q, kv):
    """Gather K/V page by page into contiguous fp64 tensors, then torch."""
    P, g = w.page_size, w.hq // w.hkv
    out = torch.zeros(w.batch, w.hq, w.head_dim, dtype=torch.float64)
    lse = torch.zeros(w.batch, w.hq, dtype=torch.float64)
    for i in range(w.batch):
        pages = t["indices"][t["indptr"][i]:t["indptr"][i + 1]]
        ks, vs = [], []
        for n, pg in enumerate(pages):
            valid = P if n < len(pages) - 1 else int(t["last"][i])
            ks.append(kv[int(pg), 0, :valid])      # [valid, Hkv, D]
            vs.append(kv[int(pg), 1, :valid])
        K = torch.cat(ks).double()
        V = torch.cat(vs).double()
        for h in range(w.hq):
            qq = q[i, h].double()
            s = (K[:, h // g, :] @ qq) / math.sqrt(w.head_dim)
            out[i, h] = torch.softmax(s, dim=0) @ V[:, h // g, :]
            lse[i, h] = torch.logsumexp(s, dim=0)
    return out.numpy(), lse.numpy()


@pytest.mark.parametrize("P,lens,hq,hkv", [
    (16, [37, 16, 5], 8, 2),
    (4, [1, 9, 12, 3], 4, 4),
    (1, [7, 1, 13], 8, 1),
    (3, [10, 3, 4], 6, 3),
])
def test_brute_force_dense(P, lens, hq, hkv):
    w, t, q, kv = _tiny(7 + P, lens, P, hq, hkv)
    ref_o, ref_l = _dense_reference(w, t, q, kv)
    o, l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=hq, hkv=hkv)
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, ref_l, rtol=0, atol=1e-12)


def _to_hnd(kv):
    """[pages, 2, P, Hkv, D] -> [pages, 2, Hkv, P, D] by explicit element
    moves (no library permute), for tiny caches."""
    pages, two, P, hkv, D = kv.shape
    out = torch.empty(pages, two, hkv, P, D, dtype=kv.dtype)
    for pg in range(pages):
        for c in range(two):
            for s in range(P):
                for h in range(hkv):
                    out[pg, c, h, s, :] = kv[pg, c, s, h, :]
    return out


@pytest.mark.parametrize("P,lens,hq,hkv", [
    (16, [37, 16, 5], 8, 2),
    (4, [1, 9, 12, 3], 4, 4),
    (3, [10, 3, 4], 6, 3),
])
def test_brute_force_dense_hnd(P, lens, hq, hkv):
    """HND cache ("FlashInfer 完全拆解", 接口层最容易踩的四个坑: the last three
    dimensions ordered head, token, dim): the oracle reading the HND copy
    equals the dense reference gathered from the NHD original."""
    w, t, q, kv = _tiny(17 + P, lens, P, hq, hkv)
    ref_o, ref_l = _dense_reference(w, t, q, kv)
    o, l = oracle.decode(q, _to_hnd(kv), t["indptr"], t["indices"], t["last"], hq=hq, hkv=hkv,
                         layout="HND")
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, ref_l, rtol=0, atol=1e-12)
    # the same bytes read with the NHD strides give a different answer, so the
    # check above does see the layout
    if hkv > 1 and P > 1:
        bad = _to_hnd(kv).reshape(kv.shape)
        o2, _ = oracle.decode(q, bad, t["indptr"], t["indices"], t["last"], hq=hq, hkv=hkv)
        assert np.abs(o2 - ref_o).max() > 1e-3


def test_fp8_hnd_equals_nhd():
    w, t, q, _ = _tiny(29, [33, 7, 50], 16, 8, 2)
    kv8, scale = workloads.make_kv_fp8(w)
    kv8 = kv8[0]
    a = oracle.decode_fp8(q, kv8, t["indptr"], t["indices"], t["last"], hq=8, hkv=2,
                          k_scale=scale, v_scale=2 * scale)
    hnd = _to_hnd(kv8.view(torch.uint8)).view(torch.float8_e4m3fn)
    b = oracle.decode_fp8(q, hnd, t["indptr"], t["indices"], t["last"], hq=8, hkv=2,
                          k_scale=scale, v_scale=2 * scale, layout="HND")
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_peaky_scores_brute_force():
    w, t, q, kv = _tiny(3, [40, 17], 16, 4, 2, scale_q=8.0)
    ref_o, ref_l = _dense_reference(w, t, q, kv)
    o, l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=4, hkv=2)
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-11)
    np.testing.assert_allclose(l, ref_l, rtol=1e-13, atol=1e-11)


def test_single_token_closed_form():
    w, t, q, kv = _tiny(11, [1, 1], 16, 4, 2)
    o, l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=4, hkv=2)
    for i in range(2):
        pg = int(t["indices"][t["indptr"][i]])
        for h in range(4):
            k = kv[pg, 0, 0, h // 2].double()
            v = kv[pg, 1, 0, h // 2].double()
            np.testing.assert_array_equal(o[i, h], v.numpy())
            s = float(q[i, h].double() @ k) / math.sqrt(w.head_dim)
            assert abs(l[i, h] - s) < 1e-12


def test_identical_keys_closed_form():
    w, t, q, kv = _tiny(12, [21], 4, 2, 1)
    kv = kv.clone()
    kv[:, 0] = kv[int(t["indices"][0]), 0, 0]      # every key equals one key
    o, l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=2, hkv=1)
    pages = t["indices"][t["indptr"][0]:t["indptr"][1]]
    vs = [kv[int(pg), 1, :(4 if n < len(pages) - 1 else int(t["last"][0]))]
          for n, pg in enumerate(pages)]
    V = torch.cat(vs).double()[:, 0, :]
    k = kv[int(t["indices"][0]), 0, 0, 0].double()
    for h in range(2):
        np.testing.assert_allclose(o[0, h], V.mean(0).numpy(), atol=1e-12)
        s = float(q[0, h].double() @ k) / math.sqrt(w.head_dim)
        assert abs(l[0, h] - (s + math.log(21))) < 1e-12


def test_gqa_grouping_is_consecutive():
    """Query head h reads KV head h // g: with distinct KV heads a wrong
    grouping (e.g. h % Hkv) gives different numbers."""
    w, t, q, kv = _tiny(13, [9], 16, 4, 2)
    q = q.clone()
    q[0, 1] = q[0, 0]
    q[0, 2] = q[0, 0]
    o, _ = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=4, hkv=2)
    np.testing.assert_array_equal(o[0, 0], o[0, 1])      # same group
    assert np.abs(o[0, 0] - o[0, 2]).max() > 1e-3         # other group


# ------------------------------------------------------------- merge algebra

def _chunk_states(q, kv, t, req, head, cuts, hq, hkv):
    rows = [(req, head, a, b) for a, b in zip(cuts[:-1], cuts[1:])]
    return oracle.attend(q, kv, t["indptr"], t["indices"], t["last"], rows,
                         hq=hq, hkv=hkv)


def test_merge_of_chunks_equals_unsplit():
    w, t, q, kv = _tiny(21, [40, 33], 4, 4, 2)
    for req, head in [(0, 0), (0, 3), (1, 2)]:
        L = w.lens[req]
        full_o, full_l = oracle.attend(q, kv, t["indptr"], t["indices"], t["last"],
                                       [(req, head)], hq=4, hkv=2)
        cuts = [0, 13, 29, L] if L > 29 else [0, 7, 19, L]
        co, cl = _chunk_states(q, kv, t, req, head, cuts, 4, 2)
        # left fold in chunk order
        o, l = co[0:1], cl[0:1]
        for k in range(1, len(co)):
            o, l = oracle.merge(o, l, co[k:k + 1], cl[k:k + 1])
        np.testing.assert_allclose(o, full_o, atol=1e-12)
        np.testing.assert_allclose(l, full_l, atol=1e-12)
        # every order and both associations give the same state
        for perm in itertools.permutations(range(3)):
            a, b, c = (co[p:p + 1] for p in perm)
            la, lb, lc = (cl[p:p + 1] for p in perm)
            o1, l1 = oracle.merge(*oracle.merge(a, la, b, lb), c, lc)
            o2, l2 = oracle.merge(a, la, *oracle.merge(b, lb, c, lc))
            np.testing.assert_allclose(o1, full_o, atol=1e-12)
            np.testing.assert_allclose(o2, full_o, atol=1e-12)
            np.testing.assert_allclose(l1, full_l, atol=1e-12)
            np.testing.assert_allclose(l2, full_l, atol=1e-12)


def test_merge_empty_state_and_closed_forms():
    rng = np.random.default_rng(0)
    o = rng.standard_normal((5, 8))
    l = rng.standard_normal(5)
    empty_o = rng.standard_normal((5, 8))
    empty_l = np.full(5, -np.inf)
    mo, ml = oracle.merge(o, l, empty_o, empty_l)
    np.testing.assert_array_equal(mo, o)
    np.testing.assert_array_equal(ml, l)
    mo, ml = oracle.merge(empty_o, empty_l, o, l)
    np.testing.assert_array_equal(mo, o)
    # both empty: zero output, empty state
    mo, ml = oracle.merge(empty_o, empty_l, empty_o, empty_l)
    assert np.all(mo == 0) and np.all(np.isneginf(ml))
    # equal lse: plain average, lse + ln 2
    o2 = rng.standard_normal((5, 8))
    mo, ml = oracle.merge(o, l, o2, l)
    np.testing.assert_allclose(mo, (o + o2) / 2, atol=1e-15)
    np.testing.assert_allclose(ml, l + math.log(2), atol=1e-15)
    # weights follow exp(lse): lse_b = lse_a + ln 3 -> weights 1/4, 3/4
    mo, ml = oracle.merge(o, l, o2, l + math.log(3))
    np.testing.assert_allclose(mo, 0.25 * o + 0.75 * o2, atol=1e-14)
    np.testing.assert_allclose(ml, l + math.log(4), atol=1e-14)


# ------------------------------------------------------------ plan restatement

def _check_plan_case(case):
    P = case["page_size"]
    indptr, indices, last = workloads.page_table(case["kv_lens"], P)
    p = oplan.plan(indptr, indices, last, page_size=P, num_pages=int(indptr[-1]),
                   n_cta=case["n_cta"], alpha=case["alpha"],
                   min_chunk_tokens=case["min_chunk_tokens"])
    assert p.chunk == case["chunk"]
    assert p.makespan == case["makespan"]
    assert p.cta_indptr == case["cta_indptr"]
    assert [list(x) for x in p.items] == case["items"]
    assert [list(x) for x in p.units] == case["units"]
    assert p.merge_indptr == case["merge_indptr"]
    if case.get("page_list_is_identity"):
        assert p.page_list == list(range(int(indptr[-1])))
    else:
        assert p.page_list == case["page_list"]


@pytest.mark.parametrize("idx", [0, 1])
def test_plan_hand_worked(idx):
    _check_plan_case(_golden("plan_hand.json")["cases"][idx])


def coverage_check(p, indptr, indices, last, page_size, group_indptr=None):
    """Independent check of a schedule: every (request, token of its table
    row) covered exactly once, page references consistent with the table,
    partial slots of each split request contiguous in chunk order, split
    requests listed longest first."""
    P = page_size
    n_rows = len(last)
    row_lens = [P * (indptr[i + 1] - indptr[i] - 1) + last[i] for i in range(n_rows)]
    if group_indptr is None:
        req_row = list(range(n_rows))
    else:
        req_row = [j for j in range(n_rows) for _ in range(group_indptr[j], group_indptr[j + 1])]
    seen = [np.zeros(row_lens[req_row[r]], dtype=np.int32) for r in range(len(req_row))]
    slots_of = {}
    for (r0, tb, te, dst, fp, n, stride) in p.items:
        row = req_row[r0]
        assert n >= 1 and all(req_row[r] == row for r in range(r0, r0 + n))
        assert 0 <= tb < te <= row_lens[row] and tb % P == 0
        assert fp == indptr[row] + tb // P
        for t in range(tb, te):
            assert p.page_list[fp + (t - tb) // P] == indices[indptr[row] + t // P]
        for i in range(n):
            seen[r0 + i][tb:te] += 1
            if dst >= 0:
                slots_of.setdefault(r0 + i, []).append((tb, dst + i * stride))
    for s_ in seen:
        assert np.all(s_ == 1)
    assert p.cta_indptr[0] == 0 and p.cta_indptr[-1] == len(p.items)
    assert all(a <= b for a, b in zip(p.cta_indptr, p.cta_indptr[1:]))
    for u, (req, nc) in enumerate(p.units):
        got = sorted(slots_of[req])
        assert [d for _, d in got] == list(range(p.merge_indptr[u], p.merge_indptr[u + 1]))
        assert nc == len(got) >= 2
    assert set(slots_of) == {r for r, _ in p.units}
    # units longest first (most chunks), ties by ascending request
    assert p.units == sorted(p.units, key=lambda u: (-u[1], u[0]))


@pytest.mark.parametrize("seed", range(6))
def test_plan_coverage_random(seed):
    rng = np.random.default_rng(seed)
    P = int(rng.choice([1, 2, 16]))
    B = int(rng.integers(1, 40))
    lens = rng.integers(1, 3000, B).tolist()
    if seed % 2:
        lens[0] = 20000
    pool = sum(-(-l // P) for l in lens) + 5
    ids = rng.permutation(pool).astype(np.int32)
    indptr, indices, last = workloads.page_table(lens, P, ids)
    n_cta = int(rng.choice([3, 16, 152]))
    p = oplan.plan(indptr, indices, last, page_size=P, num_pages=pool, n_cta=n_cta,
                   alpha=int(rng.integers(0, 64)), min_chunk_tokens=int(rng.choice([1, 64, 256])))
    coverage_check(p, indptr.tolist(), indices.tolist(), last.tolist(), P)
    W = sum(lens)
    assert len(p.items) <= B + 4 * n_cta + 4
    assert p.makespan * n_cta >= W                   # a makespan is at least the mean


@pytest.mark.parametrize("seed", range(6))
def test_grouped_plan_coverage_random(seed):
    """Shared-prefix plans: groups of requests over one table row each, cut
    into blocks of `rows` requests."""
    rng = np.random.default_rng(40 + seed)
    P = int(rng.choice([1, 16]))
    n_groups = int(rng.integers(1, 6))
    sizes = rng.integers(1, 40, n_groups).tolist()
    group_indptr = [0] + np.cumsum(sizes).tolist()
    lens = rng.integers(1, 9000, n_groups).tolist()
    pool = sum(-(-l // P) for l in lens) + 2
    indptr, indices, last = workloads.page_table(lens, P, rng.permutation(pool).astype(np.int32))
    rows = int(rng.choice([2, 4, 8, 16]))
    n_cta = int(rng.choice([5, 64, 152]))
    p = oplan.plan(indptr, indices, last, page_size=P, num_pages=pool, n_cta=n_cta, alpha=32,
                   min_chunk_tokens=256, group_indptr=group_indptr, rows=rows)
    coverage_check(p, indptr.tolist(), indices.tolist(), last.tolist(), P, group_indptr)
    assert all(n <= rows for (_, _, _, _, _, n, _) in p.items)


def test_grouped_plan_hand_worked():
    """One group of 5 requests sharing 40 tokens (P 16), blocks of 2, 3 CTAs,
    alpha 0, floor 16.  Blocks: requests {0,1}, {2,3}, {4}, each 40 tokens:
    W = 120, L = 40 -> chunk 48 (page-rounded): three whole-row items of cost
    40 (makespan 40); L/2 = 20 -> chunk 32: six items 32, 32, 32, 8, 8, 8 ->
    loads 40, 40, 40 (tie, larger chunk kept).  No split, so every item writes
    through; CTA c takes block c."""
    indptr, indices, last = workloads.page_table([40], 16)
    p = oplan.plan(indptr, indices, last, page_size=16, num_pages=3, n_cta=3, alpha=0,
                   min_chunk_tokens=16, group_indptr=[0, 5], rows=2)
    assert p.chunk == 48 and p.makespan == 40
    assert p.cta_indptr == [0, 1, 2, 3]
    assert p.items == [(0, 0, 40, -1, 0, 2, 0), (2, 0, 40, -1, 0, 2, 0), (4, 0, 40, -1, 0, 1, 0)]
    assert p.units == [] and p.merge_indptr == [0]


def test_plan_units_longest_first_hand_worked():
    """lens [40, 100], P 1, 4 CTAs, alpha 0, floor 1.  L = 35.  c = 35: items
    35 (r0), 5 (r0), 35, 35, 30 (r1); LPT order 35 r0c0, 35 r1c0, 35 r1c1,
    30 r1c2, 5 r0c1 -> CTAs 0, 1, 2, 3, then 5 onto CTA 3 (30): makespan 35.
    c = 18: seven items of 18 round-robin -> 36, 36, 36, 18; 10 and 4 onto
    CTA 3: makespan 36.  c = 9: fifteen items of 9 -> 36, 36, 36, 27; 4 and 1
    onto CTA 3: makespan 36.  So chunk 35.  Both requests are split: request
    1 has 3 chunks, request 0 has 2, so request 1 is the first unit (slots
    0..2) and request 0 the second (slots 3..4)."""
    indptr, indices, last = workloads.page_table([40, 100], 1)
    p = oplan.plan(indptr, indices, last, page_size=1, num_pages=140, n_cta=4, alpha=0,
                   min_chunk_tokens=1)
    assert p.chunk == 35 and p.makespan == 35
    assert p.units == [(1, 3), (0, 2)] and p.merge_indptr == [0, 3, 5]
    assert p.cta_indptr == [0, 1, 2, 3, 5]
    assert p.items == [(0, 0, 35, 3, 0, 1, 2), (1, 0, 35, 0, 40, 1, 3),
                       (1, 35, 70, 1, 75, 1, 3), (1, 70, 100, 2, 110, 1, 3),
                       (0, 35, 40, 4, 35, 1, 2)]
    coverage_check(p, indptr, indices, last, 1)


# ---- chunk size by search (variant of P1)

def test_search_chunk_hand_worked():
    """lens [100, 50, 30], P 16, floor 16.  Items at chunk c: c=16 -> 7+4+2 =
    13; c=32 -> 4+2+1 = 7; c=48 -> 3+2+1 = 6; c=64 -> 2+1+1 = 4; c=80, 96 ->
    4; c=112 -> 3.  Need 8 items: 16.  Need 4: 96 (the largest with 4).
    Need 3: 112 = the longest request rounded up (no split).  Need 14: even
    the floor gives 13 -> the floor."""
    lens = [100, 50, 30]
    assert oplan.search_chunk(lens, page_size=16, n_cta=8, floor=16) == 16
    assert oplan.search_chunk(lens, page_size=16, n_cta=4, floor=16) == 96
    assert oplan.search_chunk(lens, page_size=16, n_cta=3, floor=16) == 112
    assert oplan.search_chunk(lens, page_size=16, n_cta=14, floor=16) == 16
    assert oplan.search_chunk(lens, page_size=16, n_cta=4, floor=256) == 256
    assert oplan.search_chunk([], page_size=16, n_cta=4, floor=256) == 256


@pytest.mark.parametrize("seed", range(8))
def test_search_chunk_defining_property(seed):
    """The chosen chunk c fills the GPU (>= n_cta items) and c + P does not,
    unless c is the floor or the longest request (no split)."""
    rng = np.random.default_rng(70 + seed)
    P = int(rng.choice([1, 4, 16]))
    lens = rng.integers(1, 5000, int(rng.integers(1, 60))).tolist()
    n_cta = int(rng.choice([4, 37, 152]))
    floor = P * int(rng.integers(1, 20))
    c = oplan.search_chunk(lens, page_size=P, n_cta=n_cta, floor=floor)
    assert c % P == 0 and c >= floor
    top = max(-(-max(lens) // P) * P, floor)
    if c == floor:
        assert oplan.n_split_items(lens, c) < n_cta or c == top or \
            oplan.n_split_items(lens, c + P) < n_cta
    else:
        assert oplan.n_split_items(lens, c) >= n_cta
        assert c == top or oplan.n_split_items(lens, c + P) < n_cta
    # brute force over every page multiple
    ok = [k for k in range(floor, top + 1, P) if oplan.n_split_items(lens, k) >= n_cta]
    assert c == (max(ok) if ok else floor)


@pytest.mark.parametrize("seed", range(4))
def test_search_rule_plan_coverage(seed):
    rng = np.random.default_rng(90 + seed)
    P = int(rng.choice([1, 16]))
    lens = rng.integers(1, 6000, int(rng.integers(1, 50))).tolist()
    if seed % 2:
        lens[-1] = 30000
    pool = sum(-(-l // P) for l in lens) + 2
    indptr, indices, last = workloads.page_table(lens, P, rng.permutation(pool).astype(np.int32))
    n_cta = int(rng.choice([8, 152]))
    p = oplan.plan(indptr, indices, last, page_size=P, num_pages=pool, n_cta=n_cta, alpha=32,
                   min_chunk_tokens=256, chunk_rule="search")
    coverage_check(p, indptr.tolist(), indices.tolist(), last.tolist(), P)
    floor = -(-256 // P) * P
    assert p.chunk == oplan.search_chunk(lens, page_size=P, n_cta=n_cta, floor=floor)
    assert len(p.items) <= len(lens) + 4 * n_cta + 8


def test_per_head_plan_hand_worked():
    """Dense-prefix (per-head) plan: one group of 3 requests sharing 40 tokens
    (P 16), Hkv 2, 2 CTAs, alpha 0, floor 16, blocks of 32 requests.  Units
    (block 0, head 0) and (block 0, head 1), 40 tokens each: W = 80, L = 40 ->
    chunk 48: one 40-token item per unit, one per CTA (makespan 40); the
    chunks 32 and 16 also give 40 (ties keep the larger chunk)."""
    indptr, indices, last = workloads.page_table([40], 16)
    p = oplan.plan(indptr, indices, last, page_size=16, num_pages=3, n_cta=2, alpha=0,
                   min_chunk_tokens=16, group_indptr=[0, 3], rows=32, per_head=2)
    assert p.chunk == 48 and p.makespan == 40
    assert p.cta_indptr == [0, 1, 2]
    assert p.items == [(0, 0, 40, -1, 0, 3, 0), (0, 0, 40, -1, 0, 3, 0)]
    assert p.heads == [0, 1]
    assert p.units == [] and p.merge_indptr == [0]


# ---- cascade plans (shared prefix + suffixes in one schedule)

def cascade_coverage_check(p, group_indptr, prefix, suffix, P, hkv):
    """Independent check of a cascade schedule: for every request and KV
    head, each token of its group's prefix and of its own suffix is covered
    exactly once; page references agree with the two tables; each request's
    slots merge_indptr[r] .. merge_indptr[r+1] are written exactly once per
    KV head (prefix chunks first, then suffix chunks); CTAs [0, n_pre) hold
    only prefix items."""
    p_ip, p_ix, p_last = [list(map(int, x)) for x in prefix]
    s_ip, s_ix, s_last = [list(map(int, x)) for x in suffix]
    gi = list(map(int, group_indptr))
    batch = gi[-1]
    group_of = [j for j in range(len(gi) - 1) for _ in range(gi[j], gi[j + 1])]
    plen = [P * (p_ip[j + 1] - p_ip[j] - 1) + p_last[j] for j in range(len(p_last))]
    slen = [P * (s_ip[r + 1] - s_ip[r] - 1) + s_last[r] for r in range(batch)]
    nnz_p = p_ip[-1]
    pre_seen = [np.zeros((hkv, plen[group_of[r]]), np.int32) for r in range(batch)]
    suf_seen = [np.zeros(slen[r], np.int32) for r in range(batch)]
    slot_seen = [np.zeros((hkv, p.merge_indptr[r + 1] - p.merge_indptr[r]), np.int32)
                 for r in range(batch)]
    n_pre_items = p.cta_indptr[p.n_pre]
    for idx, (r0, tb, te, dst, fp, n, stride, head) in enumerate(p.items):
        assert tb % P == 0 and tb < te
        if idx < n_pre_items:
            assert stride == -1 and 0 <= head < hkv
            j = group_of[r0]
            assert all(group_of[r] == j for r in range(r0, r0 + n)) and te <= plen[j]
            assert fp == p_ip[j] + tb // P
            for t in range(tb, te):
                assert p.page_list[fp + (t - tb) // P] == p_ix[p_ip[j] + t // P]
            for r in range(r0, r0 + n):
                pre_seen[r][head, tb:te] += 1
                slot_seen[r][head, dst] += 1
        else:
            assert n == 1 and stride == 0 and head == 0 and te <= slen[r0]
            assert fp == nnz_p + s_ip[r0] + tb // P
            for t in range(tb, te):
                assert p.page_list[fp + (t - tb) // P] == s_ix[s_ip[r0] + t // P]
            suf_seen[r0][tb:te] += 1
            slot_seen[r0][:, dst - p.merge_indptr[r0]] += 1
    for r in range(batch):
        assert np.all(pre_seen[r] == 1) and np.all(suf_seen[r] == 1)
        assert np.all(slot_seen[r] == 1)
        assert p.units[r] == (r, p.merge_indptr[r + 1] - p.merge_indptr[r])
    assert p.cta_indptr[0] == 0 and p.cta_indptr[-1] == len(p.items)
    assert all(a <= b for a, b in zip(p.cta_indptr, p.cta_indptr[1:]))


def test_cascade_plan_hand_worked():
    """One group of 2 requests sharing 32 tokens, suffixes of 5 and 20 tokens
    (P 16, Hkv 1, blocks of 2), 3 CTAs, alpha 0, prefix alpha 0, prefix cost
    16/16 (a prefix token costs a suffix token), both floors 16.
    One unit (1 block x 1 head) fits the grid, so budgets are 1 + j (j <= 1).
    Costs: prefix 32 x 16 = 512, suffix 25 x 16 = 400 -> proportional
    (3 x 512 + 456) // 912 = 2 CTAs -> j = 1.  Budget 2: the block starts at
    chunk 32, one more CTA gives it chunk 16 (not below the floor): two
    items of 16 on CTAs 0 and 1 (span 16); the suffix on the 1 CTA left:
    bound 25 -> chunk 32, items 20 and 5 (span 25; chunk 16 also gives 25,
    the larger kept) -> max(16, 25) = 25.  Budget 1 (j = 0): one prefix
    item of 32 -> 32, worse.  So n_pre = 2, makespan 25.  Request slots: 2
    prefix chunks + 1 suffix chunk each -> merge_indptr [0, 3, 6]; the suffix
    items (longest first) write slots 3 + 2 = 5 (request 1) and 0 + 2 = 2
    (request 0)."""
    prefix = workloads.page_table([32], 16)            # pages 0, 1
    suffix = workloads.page_table([5, 20], 16, np.array([2, 3, 4], np.int32))
    p = oplan.plan_cascade([0, 2], prefix, suffix, page_size=16, num_pages=5, n_cta=3, hkv=1,
                           rows=2, alpha=0, prefix_alpha=0, prefix_cost16=16, suffix_floor=16,
                           prefix_floor=16)
    assert (p.n_pre, p.chunk_pre, p.chunk_suf, p.makespan) == (2, 16, 32, 25)
    assert p.cta_indptr == [0, 1, 2, 4]
    assert p.items == [(0, 0, 16, 0, 0, 2, -1, 0), (0, 16, 32, 1, 1, 2, -1, 0),
                       (1, 0, 20, 5, 3, 1, 0, 0), (0, 0, 5, 2, 2, 1, 0, 0)]
    assert p.units == [(0, 3), (1, 3)] and p.merge_indptr == [0, 3, 6]
    assert p.page_list == [0, 1, 2, 3, 4]
    cascade_coverage_check(p, [0, 2], prefix, suffix, 16, 1)


def test_cascade_prefix_level_gives_back_idle_chunks():
    """Two blocks of 1,024 prefix tokens, one KV head, budget 5, page 16,
    floor 128, worked by hand: water-filling gives block 0 a second chunk
    (512), block 1 a second (512), block 0 a third (ceil(1024 / 3) = 342 ->
    352); the longest chunk is still 512, so block 0's third chunk shortens
    nothing and is given back: chunks 512 and 512 on 4 CTAs, span 512."""
    span, queues, chunks, used = oplan._prefix_level([1024, 1024], 1, 5, 16, 128, 0)
    assert (span, chunks, used) == (512, [512, 512], 4)
    assert [q[0][3:] for q in queues] == [(0, 512), (512, 1024), (0, 512), (512, 1024)]
    # budget 6: the third chunk of each block lowers the longest to 352
    span, _, chunks, used = oplan._prefix_level([1024, 1024], 1, 6, 16, 128, 0)
    assert (span, chunks, used) == (352, [352, 352], 6)


@pytest.mark.parametrize("seed", range(6))
def test_cascade_plan_coverage_random(seed):
    rng = np.random.default_rng(70 + seed)
    P = 16
    n_groups = int(rng.integers(1, 4))
    sizes = rng.integers(1, 70, n_groups).tolist()
    gi = [0] + np.cumsum(sizes).tolist()
    B = gi[-1]
    plens = rng.integers(1, 20000, n_groups).tolist()
    slens = rng.integers(1, 3000, B).tolist()
    pool = sum(-(-l // P) for l in plens) + sum(-(-l // P) for l in slens) + 3
    ids = rng.permutation(pool).astype(np.int32)
    n_pp = sum(-(-l // P) for l in plens)
    prefix = workloads.page_table(plens, P, ids[:n_pp])
    suffix = workloads.page_table(slens, P, ids[n_pp:])
    hkv = int(rng.choice([1, 2, 8]))
    n_cta = int(rng.choice([2, 19, 152]))
    p = oplan.plan_cascade(gi, prefix, suffix, page_size=P, num_pages=pool, n_cta=n_cta, hkv=hkv,
                           rows=int(rng.choice([16, 32, 128])), alpha=32, prefix_alpha=128,
                           prefix_cost16=2, suffix_floor=128)
    assert 1 <= p.n_pre <= n_cta - 1
    cascade_coverage_check(p, gi, prefix, suffix, P, hkv)
