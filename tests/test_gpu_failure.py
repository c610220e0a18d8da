"""Failure detection on the GPU without a fault or a hang: the kernels' waits
are bounded, and a wait that runs out comes back as a device error bit the
host reads, with the context still usable afterwards (FlashInfer, in depth,
"Failure modes in production").  The self-test kernel waits, through the
kernels' own bounded-wait helper, on barriers that nothing arrives on."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_host_gb300 as pkd
import workloads

pytestmark = pytest.mark.gpu

LIMIT_NS = 2_000_000_000   # the kernels' wait limit


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkd.build()
    pkd.load()


def _small_decode_matches_oracle():
    w = workloads.Workload("after", 5, 32, 8, 128, 16, 1, (37, 16, 5), 64)
    t = workloads.make_tables(w)
    q = workloads.make_q(w, device="cuda")[0]
    kv = workloads.make_kv(w, device="cuda")[0]
    dec = pkd.BatchDecodeWithPagedKVCache(32, 8, 128, 16, max_batch=3, max_num_pages=8,
                                          num_pages=64)
    dec.plan(t["indptr"], t["indices"], t["last"])
    out, lse = dec.run(q, kv)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode(q, kv, t["indptr"], t["indices"], t["last"], hq=32, hkv=8)
    assert np.abs(out.double().cpu().numpy() - ref_o).max() <= 2e-2
    assert np.abs(lse.double().cpu().numpy() - ref_l).max() <= 1e-3
    assert dec.device_error() == 0


def test_wait_runs_out_and_reports_timeout():
    err, ns = pkd.selftest_bounded_wait(0)
    assert err == pkd.DEV_ERR_TIMEOUT
    assert 0.95 * LIMIT_NS <= ns[0] <= 3 * LIMIT_NS
    assert ns[1] == 0
    _small_decode_matches_oracle()      # the context survived


def test_abort_flag_ends_the_other_waits():
    err, ns = pkd.selftest_bounded_wait(1)
    assert err == pkd.DEV_ERR_TIMEOUT
    assert 0.95 * LIMIT_NS <= ns[0] <= 3 * LIMIT_NS
    # the second wait started half a limit late and ended on the flag, well
    # before its own limit
    assert 0 < ns[1] <= 0.8 * LIMIT_NS
    _small_decode_matches_oracle()


def test_selftest_rejects_bad_arguments():
    lib = pkd.load()
    assert lib.pkd_selftest_bounded_wait(2, None, None, None) == -1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.pkd_selftest_bounded_wait(0, err.data_ptr(), None, None) == -1
