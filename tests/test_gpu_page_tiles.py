"""GPU parity of the page-tile producer (one TMA tensor copy per 16 tokens of
K or V, 128-byte swizzle) against the fp64 oracle, and against the token-row
producer, which must give bit-identical outputs: both deliver the same bytes
to the same consumer arithmetic.

The slots past each request's last valid token are filled with NaN: a page
tile copies them (they are in-page bytes), so the consumers must mask them
out of the scores and zero them in V."""
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


def _poison_tails(kv, t, P, nan_bits):
    """Write NaN into every slot past last_page_len of each request's last
    page (K and V), in place."""
    raw = kv.view(torch.uint8) if kv.dtype != torch.uint8 else kv
    ind, ptr, last = t["indices"], t["indptr"], t["last"]
    for i in range(len(last)):
        page = int(ind[int(ptr[i + 1]) - 1])
        if int(last[i]) < P:
            if kv.dtype == torch.bfloat16:
                kv[page, :, int(last[i]):] = float("nan")
            else:
                raw[page, :, int(last[i]):] = nan_bits


def _decoder(w, t, *, split, **kw):
    extra = dict(num_ctas=1, min_chunk_tokens=1 << 30) if split == "writethrough" else \
        dict(num_ctas=7, alpha=0, min_chunk_tokens=1)
    return pkd.BatchDecodeWithPagedKVCache(
        w.hq, w.hkv, 128, w.page_size, max_batch=w.batch,
        max_num_pages=int(t["indptr"][-1]), num_pages=w.pool_pages, **extra, **kw)


CASES = [
    # (seed, lens, P, Hq, Hkv)
    (1, [37, 16, 5], 16, 32, 8),
    (2, [1, 2, 15, 16, 17, 31, 33, 47, 100], 16, 32, 8),
    (3, [700, 41, 1, 64], 32, 16, 8),        # two boxes per page
    (4, [900, 260, 35], 48, 16, 4),          # three boxes per page, 4 KV heads
    (5, [450, 18, 129], 64, 4, 2),           # 2 KV heads, g = 2
    (6, [333, 5, 64], 16, 8, 1),             # MQA, g = 8
    (7, [1200, 3], 16, 8, 8),                # g = 1
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{c[0]}" for c in CASES])
@pytest.mark.parametrize("split", ["writethrough", "split"])
def test_bf16_page_tiles_parity_and_rows_identical(case, split):
    seed, lens, P, hq, hkv = case
    w = workloads.Workload(f"t{seed}", 200 + seed, hq, hkv, 128, P, 1, tuple(lens),
                           sum(-(-l // P) for l in lens) + 3)
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    ref_o, ref_l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=hq, hkv=hkv)
    _poison_tails(kv, t, P, None)
    tiles = _decoder(w, t, split=split)
    rows = _decoder(w, t, split=split, row_copies=True)
    for d in (tiles, rows):
        d.plan(t["indptr"], t["indices"], t["last"])
    assert tiles.plan_info()["page_tiles"] == 1
    assert rows.plan_info()["page_tiles"] == 0
    o1, l1 = tiles.run(q, kv)
    o2, l2 = rows.run(q, kv)
    torch.cuda.synchronize()
    _check(o1, l1, ref_o, ref_l)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert tiles.device_error() == 0 and rows.device_error() == 0


FP8_CASES = [
    (1, [37, 16, 5], 16, 32, 8),
    (2, [1, 2, 15, 16, 17, 31, 33, 47, 900], 16, 32, 8),   # stages with one box
    (3, [700, 41, 1, 64], 32, 16, 8),
    (4, [450, 18, 129], 64, 4, 2),
]


@pytest.mark.parametrize("case", FP8_CASES, ids=[f"case{c[0]}" for c in FP8_CASES])
@pytest.mark.parametrize("split", ["writethrough", "split"])
def test_fp8_page_tiles_parity_and_rows_identical(case, split):
    seed, lens, P, hq, hkv = case
    w = workloads.Workload(f"tf{seed}", 300 + seed, hq, hkv, 128, P, 1, tuple(lens),
                           sum(-(-l // P) for l in lens) + 3)
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kvs, scale = workloads.make_kv_fp8(w, device="cuda")
    kv = kvs[0]
    ks, vs = scale, scale * 0.75
    ref_o, ref_l = oracle.decode_fp8(q, kv, t["indptr"], t["indices"], t["last"], hq=hq,
                                     hkv=hkv, k_scale=ks, v_scale=vs)
    _poison_tails(kv, t, P, 0x7F)   # e4m3 NaN
    tiles = _decoder(w, t, split=split, kv_dtype="e4m3")
    rows = _decoder(w, t, split=split, kv_dtype="e4m3", row_copies=True)
    for d in (tiles, rows):
        d.plan(t["indptr"], t["indices"], t["last"])
    assert tiles.plan_info()["page_tiles"] == 1
    assert rows.plan_info()["page_tiles"] == 0
    o1, l1 = tiles.run(q, kv, k_scale=ks, v_scale=vs)
    o2, l2 = rows.run(q, kv, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    _check(o1, l1, ref_o, ref_l)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert tiles.device_error() == 0 and rows.device_error() == 0


@pytest.mark.parametrize("P", [16, 32])
def test_shared_prefix_block_page_tiles(P):
    """Row-block (shared-prefix) consumer: groups of requests over ragged
    shared tables, page tiles against the oracle and identical to rows."""
    sizes, glens, hq, hkv = [5, 3, 9], [700, 33, 2047], 32, 8
    rng = np.random.default_rng(9)
    B = sum(sizes)
    group_indptr = np.array([0] + np.cumsum(sizes).tolist(), np.int32)
    pool = sum(-(-l // P) for l in glens) + 3
    indptr, indices, last = workloads.page_table(glens, P, rng.permutation(pool).astype(np.int32))
    w = workloads.Workload(f"spt{P}", 400 + P, hq, hkv, 128, P, 1, tuple([1] * B), pool)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    # per-request expansion for the oracle
    e_ip, e_ix, e_last = [0], [], []
    for j in range(len(sizes)):
        for _ in range(sizes[j]):
            e_ix.extend(indices[indptr[j]:indptr[j + 1]].tolist())
            e_ip.append(len(e_ix))
            e_last.append(int(last[j]))
    ref_o, ref_l = oracle.decode(q, kv, np.array(e_ip, np.int32), np.array(e_ix, np.int32),
                                 np.array(e_last, np.int32), hq=hq, hkv=hkv)
    _poison_tails(kv, {"indices": indices, "indptr": indptr, "last": last}, P, None)
    res = []
    for row_copies in (False, True):
        d = pkd.BatchDecodeWithPagedKVCache(hq, hkv, 128, P, max_batch=B,
                                            max_num_pages=int(indptr[-1]), num_pages=pool,
                                            num_ctas=7, shared_prefix=True, row_copies=row_copies)
        d.plan_shared(group_indptr, indptr, indices, last)
        assert d.plan_info()["page_tiles"] == (0 if row_copies else 1)
        res.append(d.run(q, kv))
        assert d.device_error() == 0
    torch.cuda.synchronize()
    _check(res[0][0], res[0][1], ref_o, ref_l)
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])


@pytest.mark.parametrize("P,flags,tiles", [
    (16, {}, 1), (32, {}, 1), (64, {}, 1), (8, {}, 0), (3, {}, 0), (1, {}, 0),
    (16, {"row_copies": True}, 0), (16, {"use_tensor_cores": False}, 0),
    (16, {"kv_dtype": "e4m3"}, 1), (16, {"shared_prefix": True}, 1),
])
def test_producer_selection(P, flags, tiles):
    d = pkd.BatchDecodeWithPagedKVCache(32, 8, 128, P, max_batch=2, max_num_pages=8,
                                        num_pages=8, **flags)
    ind = np.array([0, 1], dtype=np.int32)
    if flags.get("shared_prefix"):
        d.plan_shared(np.array([0, 1], dtype=np.int32), np.array([0, 1], dtype=np.int32), ind[:1],
                      np.array([1], dtype=np.int32))
    else:
        d.plan(np.array([0, 1], dtype=np.int32), ind[:1], np.array([1], dtype=np.int32))
    assert d.plan_info()["page_tiles"] == tiles
