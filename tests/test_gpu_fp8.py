"""GPU parity of the FP8-E4M3 cache path against the fp64 oracle (which
decodes E4M3 from the format definition): 2e-2 on bf16 out, 1e-3 on lse."""
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


def _check(out, lse, ref_o, ref_l, rows=None):
    o = out.double().cpu().numpy()
    l = lse.double().cpu().numpy()
    if rows is not None:
        o = o[rows[:, 0], rows[:, 1]]
        l = l[rows[:, 0], rows[:, 1]]
    assert np.isfinite(o).all() and np.isfinite(l).all()
    assert np.abs(o - ref_o).max() <= OUT_TOL, np.abs(o - ref_o).max()
    assert np.abs(l - ref_l).max() <= LSE_TOL, np.abs(l - ref_l).max()


CASES = [
    (1, [37, 16, 5], 16, 32, 8),
    (2, [1, 2, 15, 16, 17, 31, 33, 900], 16, 32, 8),
    (3, [300, 7, 1024, 5], 1, 64, 8),
    (4, [513, 97, 2000], 3, 8, 8),
    (5, [450, 18], 8, 4, 2),
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{c[0]}" for c in CASES])
@pytest.mark.parametrize("split", ["writethrough", "split"])
def test_fp8_parity_every_element(case, split):
    seed, lens, P, hq, hkv = case
    w = workloads.Workload(f"f{seed}", 70 + seed, hq, hkv, 128, P, 1, tuple(lens),
                           sum(-(-l // P) for l in lens) + 5)
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kvs, scale = workloads.make_kv_fp8(w, device="cuda")
    kv = kvs[0]
    ks, vs = scale, scale * 1.5
    kw = dict(num_ctas=1, min_chunk_tokens=1 << 30) if split == "writethrough" else \
        dict(num_ctas=5, alpha=0, min_chunk_tokens=1)
    dec = pkd.BatchDecodeWithPagedKVCache(hq, hkv, 128, P, max_batch=w.batch,
                                          max_num_pages=int(t["indptr"][-1]),
                                          num_pages=w.pool_pages, kv_dtype="e4m3", **kw)
    dec.plan(t["indptr"], t["indices"], t["last"])
    out, lse = dec.run(q, kv, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode_fp8(q, kv, t["indptr"], t["indices"], t["last"], hq=hq, hkv=hkv,
                                     k_scale=ks, v_scale=vs)
    _check(out, lse, ref_o, ref_l)
    assert dec.device_error() == 0


def test_fp8_llama_step_graph_full():
    """The Llama-shaped step with an E4M3 cache, 4 layers, graph replay: every
    output of layers 0 and 3 against the oracle."""
    base = workloads.workload("llama8b_step")
    w = workloads.Workload("llama8b_step_fp8", base.seed, base.hq, base.hkv, 128, 16, 4,
                           base.lens, base.pool_pages)
    t = workloads.make_tables(w)
    qs = workloads.make_q(w, device="cuda")
    kvs, scale = workloads.make_kv_fp8(w, device="cuda")
    outs = [torch.empty_like(x) for x in qs]
    lses = [torch.empty(w.batch, w.hq, dtype=torch.float32, device="cuda") for _ in qs]
    dec = pkd.BatchDecodeWithPagedKVCache(w.hq, w.hkv, 128, 16, max_batch=w.batch,
                                          max_num_pages=int(t["indptr"][-1]),
                                          num_pages=w.pool_pages, kv_dtype="e4m3")
    dec.plan(t["indptr"], t["indices"], t["last"])
    scales = [(scale, scale * (1 + l)) for l in range(w.layers)]
    g = dec.capture(qs, kvs, outs, lses, kv_scales=scales)
    g.launch()
    torch.cuda.synchronize()
    for layer in (0, 3):
        ref_o, ref_l = oracle.decode_fp8(qs[layer], kvs[layer], t["indptr"], t["indices"],
                                         t["last"], hq=w.hq, hkv=w.hkv,
                                         k_scale=scales[layer][0], v_scale=scales[layer][1])
        _check(outs[layer], lses[layer], ref_o, ref_l)
    o2, l2 = dec.run(qs[3], kvs[3], k_scale=scales[3][0], v_scale=scales[3][1])
    torch.cuda.synchronize()
    assert torch.equal(o2, outs[3]) and torch.equal(l2, lses[3])


def test_fp8_dtype_mismatch_rejected():
    dec = pkd.BatchDecodeWithPagedKVCache(32, 8, 128, 16, max_batch=2, max_num_pages=4,
                                          num_pages=4, kv_dtype="e4m3")
    dec.plan(np.array([0, 1], np.int32), np.array([0], np.int32), np.array([3], np.int32))
    q = torch.zeros(1, 32, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(TypeError):      # planned e4m3, given a bf16 cache
        dec.run(q, torch.zeros(4, 2, 16, 8, 128, dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(pkd.PkdError):   # non-finite scale
        dec.run(q, torch.zeros(4, 2, 16, 8, 128, dtype=torch.uint8, device="cuda"),
                k_scale=float("inf"))
    with pytest.raises(pkd.PkdError):   # no CUDA-core or shared-prefix FP8 variant
        pkd.BatchDecodeWithPagedKVCache(32, 8, 128, 16, max_batch=2, max_num_pages=4,
                                        num_pages=4, kv_dtype="e4m3", use_tensor_cores=False)
