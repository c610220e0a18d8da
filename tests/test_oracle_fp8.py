"""Pins for the oracle's FP8 (E4M3) path.

* the E4M3 decoder against torch's float8_e4m3fn conversion (a library
  routine) on all 256 codes, and against values fixed by the format
  (1.0 = 0x38, 448 = 0x7e, smallest subnormal 2^-9 = 0x01, NaN = 0x7f);
* attention over an E4M3 cache with power-of-two scales equals attention
  over the same values widened to bf16 (exact) and pre-multiplied by the
  scales -- the scale contract: key = k_scale * K, value = v_scale * V.
"""
import numpy as np
import torch

import oracle
import workloads


def test_e4m3_decoder_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().double().numpy()
    got = np.array([oracle.e4m3_to_float(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    assert oracle.e4m3_to_float(0x38) == 1.0
    assert oracle.e4m3_to_float(0x7E) == 448.0
    assert oracle.e4m3_to_float(0x01) == 2.0 ** -9
    assert oracle.e4m3_to_float(0xB8) == -1.0


def test_fp8_attention_equals_scaled_bf16():
    w = workloads.Workload("f8", 3, 8, 2, 16, 4, 1, (13, 30, 1), 14)
    t = workloads.make_tables(w)
    q = workloads.make_q(w)[0]
    kv8, _ = workloads.make_kv_fp8(w)
    kv8 = kv8[0]
    ks, vs = 0.25, 4.0                     # powers of two: exact in bf16
    kvb = kv8.float()
    kvb[:, 0] *= ks
    kvb[:, 1] *= vs
    kvb = kvb.to(torch.bfloat16)
    assert torch.equal(kvb.float()[:, 0], kv8.float()[:, 0] * ks)
    o8, l8 = oracle.decode_fp8(q, kv8, t["indptr"], t["indices"], t["last"], hq=8, hkv=2,
                               k_scale=ks, v_scale=vs)
    ob, lb = oracle.decode(q, kvb, t["indptr"], t["indices"], t["last"], hq=8, hkv=2)
    np.testing.assert_allclose(o8, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l8, lb, rtol=0, atol=1e-12)
