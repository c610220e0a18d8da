"""GPU parity of the variants: the HND cache layout (decode with both
producers, bf16 and E4M3, the shared-prefix kernel, graph replay, append) and
the binary-search chunk rule, each against the fp64 oracle; an HND run must
also give the same bits as the NHD run over the same values, since both
producers land the same bytes in shared memory."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_host_gb300 as pkd
import workloads
from oracle import append as oappend
from oracle import plan as oplan

pytestmark = pytest.mark.gpu

OUT_TOL = 2e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkd.build()
    pkd.load()


def _check(out, lse, ref_o, ref_l, rows=None):
    o = out.double().cpu().numpy()
    l = lse.double().cpu().numpy()
    if rows is not None:
        o = o[rows[:, 0], rows[:, 1]]
        l = l[rows[:, 0], rows[:, 1]]
    assert np.isfinite(o).all() and np.isfinite(l).all()
    assert np.abs(o - ref_o).max() <= OUT_TOL, np.abs(o - ref_o).max()
    assert np.abs(l - ref_l).max() <= LSE_TOL, np.abs(l - ref_l).max()


def _hnd(x):
    return x.permute(0, 1, 3, 2, 4).contiguous()


def _dec(w, t, layout, *, split, **kw):
    extra = dict(num_ctas=1, min_chunk_tokens=1 << 30) if split == "writethrough" else \
        dict(num_ctas=6, alpha=0, min_chunk_tokens=1)
    return pkd.BatchDecodeWithPagedKVCache(
        w.hq, w.hkv, 128, w.page_size, max_batch=w.batch,
        max_num_pages=int(t["indptr"][-1]), num_pages=w.pool_pages, kv_layout=layout,
        **extra, **kw)


HND_CASES = [
    # (seed, lens, P, Hq, Hkv, tiles)
    (1, [37, 16, 5], 16, 32, 8, 1),
    (2, [700, 41, 1, 64], 32, 16, 8, 1),
    (3, [450, 18, 129], 8, 8, 2, 0),        # token rows, one copy per token and head
    (4, [513, 97, 200], 3, 8, 8, 0),
    (5, [300, 7, 1024, 5], 1, 64, 8, 0),    # P = 1: HND and NHD are the same bytes
]


@pytest.mark.parametrize("case", HND_CASES, ids=[f"case{c[0]}" for c in HND_CASES])
@pytest.mark.parametrize("split", ["writethrough", "split"])
def test_hnd_bf16_parity_and_same_bits_as_nhd(case, split):
    seed, lens, P, hq, hkv, tiles = case
    w = workloads.Workload(f"h{seed}", 500 + seed, hq, hkv, 128, P, 1, tuple(lens),
                           sum(-(-l // P) for l in lens) + 3)
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    kv_h = _hnd(kv)
    ref_o, ref_l = oracle.decode(q, kv_h, t["indptr"], t["indices"], t["last"], hq=hq, hkv=hkv,
                                 layout="HND")
    dh = _dec(w, t, "HND", split=split)
    dn = _dec(w, t, "NHD", split=split)
    for d in (dh, dn):
        d.plan(t["indptr"], t["indices"], t["last"])
    assert dh.plan_info()["page_tiles"] == tiles
    oh, lh = dh.run(q, kv_h)
    on, ln = dn.run(q, kv)
    torch.cuda.synchronize()
    _check(oh, lh, ref_o, ref_l)
    assert torch.equal(oh, on) and torch.equal(lh, ln)
    assert dh.device_error() == 0


@pytest.mark.parametrize("P,row_copies", [(16, False), (16, True), (8, False)])
def test_hnd_fp8_parity_and_same_bits_as_nhd(P, row_copies):
    lens, hq, hkv = [1, 15, 17, 33, 47, 900, 260], 32, 8
    w = workloads.Workload(f"hf{P}", 600 + P, hq, hkv, 128, P, 1, tuple(lens),
                           sum(-(-l // P) for l in lens) + 3)
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kvs, scale = workloads.make_kv_fp8(w, device="cuda")
    kv = kvs[0]
    kv_h = _hnd(kv.view(torch.uint8)).view(torch.float8_e4m3fn)
    ks, vs = scale, 0.5 * scale
    ref_o, ref_l = oracle.decode_fp8(q, kv_h, t["indptr"], t["indices"], t["last"], hq=hq,
                                     hkv=hkv, k_scale=ks, v_scale=vs, layout="HND")
    dh = _dec(w, t, "HND", split="split", kv_dtype="e4m3", row_copies=row_copies)
    dn = _dec(w, t, "NHD", split="split", kv_dtype="e4m3", row_copies=row_copies)
    for d in (dh, dn):
        d.plan(t["indptr"], t["indices"], t["last"])
    oh, lh = dh.run(q, kv_h, k_scale=ks, v_scale=vs)
    on, ln = dn.run(q, kv, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    _check(oh, lh, ref_o, ref_l)
    assert torch.equal(oh, on) and torch.equal(lh, ln)


def test_hnd_fma_consumer_parity():
    lens, P, hq, hkv = [333, 5, 64, 1000], 16, 32, 8
    w = workloads.Workload("hfma", 650, hq, hkv, 128, P, 1, tuple(lens),
                           sum(-(-l // P) for l in lens) + 3)
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kv_h = _hnd(workloads.make_kv(w, device="cuda")[0])
    d = _dec(w, t, "HND", split="split", use_tensor_cores=False)
    d.plan(t["indptr"], t["indices"], t["last"])
    assert d.plan_info()["page_tiles"] == 0
    o, l = d.run(q, kv_h)
    ref_o, ref_l = oracle.decode(q, kv_h, t["indptr"], t["indices"], t["last"], hq=hq, hkv=hkv,
                                 layout="HND")
    _check(o, l, ref_o, ref_l)


def test_hnd_shared_prefix_block():
    sizes, glens, P, hq, hkv = [5, 3, 9], [700, 33, 2047], 16, 32, 8
    rng = np.random.default_rng(12)
    B = sum(sizes)
    group_indptr = np.array([0] + np.cumsum(sizes).tolist(), np.int32)
    pool = sum(-(-l // P) for l in glens) + 3
    indptr, indices, last = workloads.page_table(glens, P, rng.permutation(pool).astype(np.int32))
    w = workloads.Workload("hsp", 660, hq, hkv, 128, P, 1, tuple([1] * B), pool)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    kv_h = _hnd(kv)
    e_ip, e_ix, e_last = [0], [], []
    for j in range(len(sizes)):
        for _ in range(sizes[j]):
            e_ix.extend(indices[indptr[j]:indptr[j + 1]].tolist())
            e_ip.append(len(e_ix))
            e_last.append(int(last[j]))
    ref_o, ref_l = oracle.decode(q, kv_h, np.array(e_ip, np.int32), np.array(e_ix, np.int32),
                                 np.array(e_last, np.int32), hq=hq, hkv=hkv, layout="HND")
    res = []
    for layout, cache in (("HND", kv_h), ("NHD", kv)):
        d = pkd.BatchDecodeWithPagedKVCache(hq, hkv, 128, P, max_batch=B,
                                            max_num_pages=int(indptr[-1]), num_pages=pool,
                                            num_ctas=7, shared_prefix=True, kv_layout=layout)
        d.plan_shared(group_indptr, indptr, indices, last)
        res.append(d.run(q, cache))
    torch.cuda.synchronize()
    _check(res[0][0], res[0][1], ref_o, ref_l)
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])


def test_hnd_graph_replay_full():
    """Four layers of the Llama-shaped step in HND, captured and replayed:
    every output of layers 0 and 3 against the oracle."""
    base = workloads.workload("llama8b_step_hnd")
    w = workloads.Workload(base.name, base.seed, base.hq, base.hkv, 128, 16, 4, base.lens,
                           base.pool_pages, kv_layout="HND")
    t = workloads.make_tables(w)
    qs = workloads.make_q(w, device="cuda")
    kvs = workloads.make_kv(w, device="cuda")
    outs = [torch.empty_like(x) for x in qs]
    lses = [torch.empty(w.batch, w.hq, dtype=torch.float32, device="cuda") for _ in qs]
    d = pkd.BatchDecodeWithPagedKVCache(w.hq, w.hkv, 128, 16, max_batch=w.batch,
                                        max_num_pages=int(t["indptr"][-1]),
                                        num_pages=w.pool_pages, kv_layout="HND")
    d.plan(t["indptr"], t["indices"], t["last"])
    g = d.capture(qs, kvs, outs, lses)
    d.plan(t["indptr"], t["indices"], t["last"])
    g.launch()
    torch.cuda.synchronize()
    for layer in (0, 3):
        ref_o, ref_l = oracle.decode(qs[layer], kvs[layer], t["indptr"], t["indices"], t["last"],
                                     hq=w.hq, hkv=w.hkv, layout="HND")
        _check(outs[layer], lses[layer], ref_o, ref_l)
    g.close()
    assert d.device_error() == 0


def _u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("layout,fp8", [("HND", False), ("HND", True), ("NHD", True)])
def test_append_layouts_match_oracle(layout, fp8):
    P, hkv, D = 16, 8, 128
    rng = np.random.default_rng(17 + fp8)
    lens = rng.integers(1, 300, 20).tolist()
    pool = sum(-(-l // P) for l in lens) + 5
    indptr, indices, last = workloads.page_table(lens, P, rng.permutation(pool).astype(np.int32))
    g = torch.Generator(device="cuda").manual_seed(9)
    shape = (pool, 2, hkv, P, D) if layout == "HND" else (pool, 2, P, hkv, D)
    if fp8:
        kv = torch.randint(0, 0x7F, shape, generator=g, device="cuda", dtype=torch.int32)
        kv = kv.to(torch.uint8)
    else:
        kv = torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)
    b = list(range(len(lens))) + [len(lens) + 1]
    pos = [lens[i] - 1 for i in range(len(lens))] + [0]
    n = len(b)
    if fp8:
        k_new = torch.randint(0, 0x7F, (n, hkv, D), generator=g, device="cuda",
                              dtype=torch.int32).to(torch.uint8)
        v_new = torch.randint(0, 0x7F, (n, hkv, D), generator=g, device="cuda",
                              dtype=torch.int32).to(torch.uint8)
        host = lambda x: x.cpu().numpy()
    else:
        k_new = torch.randn(n, hkv, D, generator=g, device="cuda").to(torch.bfloat16)
        v_new = torch.randn(n, hkv, D, generator=g, device="cuda").to(torch.bfloat16)
        host = _u16
    ref, skipped = oappend.append_kv(host(kv), host(k_new), host(v_new), b, pos, indptr,
                                     indices, last, P, layout=layout)
    assert skipped == [n - 1]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = lambda a: torch.tensor(np.asarray(a, dtype=np.int32), device="cuda")
    pkd.append_kv(k_new, v_new, dev(b), dev(pos), dev(indptr), dev(indices), dev(last), kv,
                  err=err, kv_layout=layout)
    torch.cuda.synchronize()
    assert np.array_equal(host(kv), ref)
    assert int(err.item()) == 2


@pytest.mark.parametrize("name", ["skewed", "llama8b_step"])
def test_search_chunk_rule_parity(name):
    """Binary-search chunk rule: the device schedule's chunk is the oracle's,
    and every output matches the oracle (full-size workload, one layer)."""
    w = workloads.workload(name)
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda", layers=1)[0]
    kv = workloads.make_kv(w, device="cuda", layers=1)[0]
    d = pkd.BatchDecodeWithPagedKVCache(w.hq, w.hkv, 128, w.page_size, max_batch=w.batch,
                                        max_num_pages=int(t["indptr"][-1]),
                                        num_pages=w.pool_pages, chunk_rule="search")
    d.plan(t["indptr"], t["indices"], t["last"])
    info = d.plan_info()
    lens = oplan.lengths(t["indptr"], t["last"], t["indices"], w.page_size, w.pool_pages)
    assert info["chunk_tokens"] == oplan.search_chunk(lens, page_size=w.page_size,
                                                      n_cta=info["num_ctas"], floor=256)
    out, lse = d.run(q, kv)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=w.hq,
                                 hkv=w.hkv)
    _check(out, lse, ref_o, ref_l)
    assert d.device_error() == 0
