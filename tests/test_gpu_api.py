"""GPU-side API contract: the failure modes the pages list (stale plan,
run before plan, dtype / layout mismatch, bad tables, workspace too small)
come back as status codes or Python exceptions before any launch; no GPU
fault is ever provoked."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_decode_host_gb300 as pkd
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkd.build()
    pkd.load()


def _setup(lens=(37, 16, 5)):
    w = workloads.Workload("api", 1, 32, 8, 128, 16, 1, tuple(lens), 64)
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    dec = pkd.BatchDecodeWithPagedKVCache(32, 8, 128, 16, max_batch=8, max_num_pages=32,
                                          num_pages=64)
    return w, t, q, kv, dec


def test_run_before_plan_and_stale_epoch():
    w, t, q, kv, dec = _setup()
    lib = pkd.load()
    out = torch.empty_like(q)
    st = lib.pkd_run(dec._h, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kv.data_ptr()),
                     ctypes.c_void_p(out.data_ptr()), None, 0, None)
    assert st == -5                                       # PKD_E_NO_PLAN
    e1 = dec.plan(t["indptr"], t["indices"], t["last"])
    e2 = dec.plan(t["indptr"], t["indices"], t["last"])
    assert e2 == e1 + 1
    with pytest.raises(pkd.PkdError) as e:
        dec.run(q, kv, expect_epoch=e1)
    assert e.value.status == -6                           # PKD_E_STALE_PLAN
    dec.run(q, kv, expect_epoch=e2)
    torch.cuda.synchronize()


def test_dtype_shape_layout_mismatch():
    w, t, q, kv, dec = _setup()
    dec.plan(t["indptr"], t["indices"], t["last"])
    with pytest.raises(TypeError):
        dec.run(q.half(), kv)                             # planned bf16, got fp16
    with pytest.raises(TypeError):
        dec.run(q, kv.half())
    with pytest.raises(ValueError):
        dec.run(q[:2].contiguous(), kv)                   # batch differs from the plan
    with pytest.raises(ValueError):
        dec.run(q, kv.transpose(2, 3).contiguous())       # HND-shaped cache, NHD plan
    with pytest.raises(ValueError):
        pkd.BatchDecodeWithPagedKVCache(32, 8, 128, 16, max_batch=8, max_num_pages=32,
                                        num_pages=64, kv_layout="NDH")
    hnd = pkd.BatchDecodeWithPagedKVCache(w.hq, w.hkv, 128, w.page_size, max_batch=w.batch,
                                          max_num_pages=int(t["indptr"][-1]),
                                          num_pages=w.pool_pages, kv_layout="HND")
    hnd.plan(t["indptr"], t["indices"], t["last"])
    with pytest.raises(ValueError):
        hnd.run(q, kv)                                    # NHD-shaped cache, HND plan


def test_bad_tables_and_capacity():
    w, t, q, kv, dec = _setup()
    for indptr, indices, last in [
        ([0, 2], [0, 1], [0]), ([0, 2], [0, 1], [17]), ([0, 0], [], [1]),
        ([0, 1], [64], [1]), ([0, 1], [-1], [1]),
    ]:
        with pytest.raises(pkd.PkdError) as e:
            dec.plan(np.array(indptr, np.int32), np.array(indices, np.int32),
                     np.array(last, np.int32))
        assert e.value.status == -2
    with pytest.raises(pkd.PkdError) as e:                # batch above capacity
        dec.plan(np.arange(10, dtype=np.int32), np.arange(9, dtype=np.int32),
                 np.ones(9, np.int32))
    assert e.value.status == -7
    with pytest.raises(TypeError):                        # int64 indices
        dec.plan(t["indptr"].astype(np.int64), t["indices"], t["last"])
    with pytest.raises(ValueError):                       # device-side table
        dec.plan(torch.tensor(t["indptr"], device="cuda"), t["indices"], t["last"])
    # a failed plan leaves the previous plan in force
    dec.plan(t["indptr"], t["indices"], t["last"])
    ep = dec.epoch
    with pytest.raises(pkd.PkdError):
        dec.plan(np.array([0, 2], np.int32), np.array([0, 1], np.int32), np.array([0], np.int32))
    assert dec.plan_info()["batch"] == 3
    dec.run(q, kv, expect_epoch=ep)
    torch.cuda.synchronize()
    assert dec.device_error() == 0


def test_workspace_too_small_and_misaligned():
    lib = pkd.load()
    cfg = pkd.make_config(32, 8, 128, 16, 64, 4096, 4096)
    need = lib.pkd_workspace_bytes(ctypes.byref(cfg))
    assert need > 0
    small = torch.empty(need // 2, dtype=torch.uint8, device="cuda")
    h = ctypes.c_void_p()
    assert lib.pkd_create(ctypes.byref(cfg), ctypes.c_void_p(small.data_ptr()), small.numel(),
                          ctypes.byref(h)) == -4
    big = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    assert lib.pkd_create(ctypes.byref(cfg), ctypes.c_void_p(big.data_ptr() + 8), need,
                          ctypes.byref(h)) == -1
    assert lib.pkd_create(ctypes.byref(cfg), ctypes.c_void_p(big.data_ptr()), need,
                          ctypes.byref(h)) == 0
    lib.pkd_destroy(h)


def test_unsupported_shapes_rejected():
    for hq, hkv, d in [(32, 8, 64), (48, 8, 128), (32, 16, 128)]:
        with pytest.raises(pkd.PkdError):
            pkd.BatchDecodeWithPagedKVCache(hq, hkv, d, 16, max_batch=4, max_num_pages=8,
                                            num_pages=8)


def test_graph_capture_with_host_io():
    """pkd_graph_capture_io: the graph copies each layer's queries in from
    page-locked host memory and its out / lse back; new host queries between
    launches give the results of direct runs on them, bit for bit."""
    layers = 3
    w = workloads.Workload("io", 7, 32, 8, 128, 16, layers, (700, 37, 1500, 5), 200)
    t = workloads.make_tables(w)
    qs_host_src = workloads.make_q(w, device="cpu")
    kvs = workloads.make_kv(w, device="cuda")
    dec = pkd.BatchDecodeWithPagedKVCache(w.hq, w.hkv, 128, 16, max_batch=w.batch,
                                          max_num_pages=int(t["indptr"][-1]),
                                          num_pages=w.pool_pages, num_ctas=9, alpha=0,
                                          min_chunk_tokens=16)
    dec.plan(t["indptr"], t["indices"], t["last"])
    assert dec.plan_info()["num_units"] >= 1           # split requests: the merge runs too
    q_dev = [torch.zeros_like(x, device="cuda") for x in qs_host_src]
    out_dev = [torch.empty_like(x) for x in q_dev]
    lse_dev = [torch.empty(w.batch, w.hq, dtype=torch.float32, device="cuda") for _ in q_dev]
    hq = [x.pin_memory() for x in qs_host_src]
    ho = [torch.zeros(x.shape, dtype=x.dtype).pin_memory() for x in q_dev]
    hl = [torch.zeros(w.batch, w.hq, dtype=torch.float32).pin_memory() for _ in q_dev]
    with pytest.raises(ValueError):                       # host buffers must be page-locked
        dec.capture(q_dev, kvs, out_dev, lse_dev, host_qs=[x.clone() for x in qs_host_src])
    g = dec.capture(q_dev, kvs, out_dev, lse_dev, host_qs=hq, host_outs=ho, host_lses=hl)
    for rnd in range(2):
        if rnd == 1:                                      # new queries, same graph
            for x in hq:
                x.copy_((x.float() * -0.5).to(torch.bfloat16))
        g.launch()
        torch.cuda.synchronize()
        for l in range(layers):
            o, s = dec.run(hq[l].cuda(), kvs[l])
            torch.cuda.synchronize()
            assert torch.equal(ho[l], o.cpu()) and torch.equal(hl[l], s.cpu())
    ref_o, ref_l = oracle_decode(hq[1], kvs[1], t, w)
    assert np.abs(ho[1].double().numpy() - ref_o).max() <= 2e-2
    assert np.abs(hl[1].double().numpy() - ref_l).max() <= 1e-3
    g.close()
    assert dec.device_error() == 0


def oracle_decode(q, kv, t, w):
    import oracle
    return oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=w.hq, hkv=w.hkv)


def test_error_poll_waits_for_its_own_stream_only():
    """pkd_last_device_error orders its read and reset on the caller's
    stream and waits for that stream alone: a long kernel on another stream
    is still running when the poll returns."""
    import time
    w, t, q, kv, dec = _setup()
    dec.plan(t["indptr"], t["indices"], t["last"])
    dec.run(q, kv)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    poll = torch.cuda.Stream()
    with torch.cuda.stream(side):
        torch.cuda._sleep(int(2e9))        # about a second of spinning at GB300 clocks
    t0 = time.perf_counter()
    err = dec.device_error(stream=poll)
    dt = time.perf_counter() - t0
    still_running = not side.query()
    side.synchronize()
    assert err == 0
    assert still_running, "the poll waited for another stream's kernel"
    assert dt < 0.25, dt


def _second_tables():
    """Another batch of three over the same 64-page pool (29 pages)."""
    w2 = workloads.Workload("api2", 2, 32, 8, 128, 16, 1, (200, 150, 90), 64)
    return w2, workloads.make_tables(w2)


def test_run_waits_on_the_device_for_a_plan_from_another_stream():
    """pkd_run with expect_epoch: the plan is uploaded on a side stream held
    back by a GPU sleep, and the run is issued on another stream with no
    event between them.  The kernels wait for the new schedule's epoch word
    and compute the new plan, not the one still in the workspace."""
    w, t, q, kv, dec = _setup()
    dec.plan(t["indptr"], t["indices"], t["last"])
    dec.run(q, kv)
    torch.cuda.synchronize()
    w2, t2 = _second_tables()
    out = torch.full_like(q, float("nan"))
    lse = torch.full((q.shape[0], q.shape[1]), float("nan"), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    side, main = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(side):
        torch.cuda._sleep(int(1e8))        # tens of milliseconds
    ep = dec.plan(t2["indptr"], t2["indices"], t2["last"], stream=side)
    dec.run(q, kv, out=out, lse=lse, expect_epoch=ep, stream=main)
    held_back = not side.query()
    torch.cuda.synchronize()
    assert held_back, "the upload had already landed when the run was issued"
    ref_o, ref_l = oracle_decode(q, kv, t2, w2)
    assert np.abs(out.double().cpu().numpy() - ref_o).max() <= 2e-2
    assert np.abs(lse.double().cpu().numpy() - ref_l).max() <= 1e-3
    assert dec.device_error() == 0


def test_device_wait_for_a_late_plan_times_out_cleanly():
    """The device-side wait for a plan's schedule is bounded: an upload held
    back past it (a GPU sleep of several seconds on its stream) makes the run
    report PKD_DEV_ERR_TIMEOUT, and the context stays usable: the same plan,
    once landed, runs correctly."""
    w, t, q, kv, dec = _setup()
    dec.plan(t["indptr"], t["indices"], t["last"])
    dec.run(q, kv)
    torch.cuda.synchronize()
    w2, t2 = _second_tables()
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    side, main = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(side):
        torch.cuda._sleep(int(1.2e10))
    ep = dec.plan(t2["indptr"], t2["indices"], t2["last"], stream=side)
    dec.run(q, kv, out=out, lse=lse, expect_epoch=ep, stream=main)
    main.synchronize()
    # the timeout bit says the wait gave up before the upload landed
    assert dec.device_error(stream=main) == pkd.DEV_ERR_TIMEOUT
    side.synchronize()
    dec.run(q, kv, out=out, lse=lse, expect_epoch=ep, stream=main)
    main.synchronize()
    ref_o, ref_l = oracle_decode(q, kv, t2, w2)
    assert np.abs(out.double().cpu().numpy() - ref_o).max() <= 2e-2
    assert np.abs(lse.double().cpu().numpy() - ref_l).max() <= 1e-3
    assert dec.device_error(stream=main) == 0
