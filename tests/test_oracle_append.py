"""Pins for the append oracle (oracle/append.py).

* hand-worked slots of the pages' worked example (lengths 37, 16, 5, page
  size 16, pages 0..4): the last token of each request lands at
  (page 2, slot 4), (page 3, slot 15), (page 4, slot 4);
* read back through the attention oracle (its own gather code): attending a
  query over the single appended token returns that token's V row, and the
  LSE is q . k / sqrt(D);
* tokens outside the table are skipped and nothing else changes.
"""
import math

import numpy as np
import torch

import oracle
import workloads
from oracle import append as oappend


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _setup(lens, P, hkv=2, D=16, pool_extra=3, seed=0):
    indptr, indices, last = workloads.page_table(lens, P)
    pages = int(indptr[-1]) + pool_extra
    g = torch.Generator().manual_seed(seed)
    kv = torch.randn(pages, 2, P, hkv, D, generator=g).to(torch.bfloat16)
    return indptr, indices, last, kv, g


def test_worked_example_slots():
    indptr, indices, last, kv, g = _setup([37, 16, 5], 16)
    n = 3
    k_new = torch.randn(n, 2, 16, generator=g).to(torch.bfloat16)
    v_new = torch.randn(n, 2, 16, generator=g).to(torch.bfloat16)
    out, skipped = oappend.append_kv(_bits(kv), _bits(k_new), _bits(v_new), [0, 1, 2],
                                     [36, 15, 4], indptr, indices, last, 16)
    assert skipped == []
    before = _bits(kv)
    expect = {(2, 4): 0, (3, 15): 1, (4, 4): 2}          # (page, slot) -> token
    for page in range(out.shape[0]):
        for slot in range(16):
            if (page, slot) in expect:
                i = expect[(page, slot)]
                np.testing.assert_array_equal(out[page, 0, slot], _bits(k_new)[i])
                np.testing.assert_array_equal(out[page, 1, slot], _bits(v_new)[i])
            else:
                np.testing.assert_array_equal(out[page, :, slot], before[page, :, slot])


def test_read_back_through_attention_oracle():
    lens, P, hkv, D = [23, 9, 40], 4, 2, 16
    indptr, indices, last, kv, g = _setup(lens, P, hkv=hkv, D=D, seed=3)
    rng = np.random.default_rng(1)
    batch_idx = [0, 1, 2, 2]
    pos = [int(rng.integers(0, lens[b])) for b in batch_idx]
    pos[3] = lens[2] - 1 if pos[2] != lens[2] - 1 else 0
    n = len(batch_idx)
    k_new = torch.randn(n, hkv, D, generator=g).to(torch.bfloat16)
    v_new = torch.randn(n, hkv, D, generator=g).to(torch.bfloat16)
    out, skipped = oappend.append_kv(_bits(kv), _bits(k_new), _bits(v_new), batch_idx, pos,
                                     indptr, indices, last, P)
    assert skipped == []
    hq = 2 * hkv
    q = torch.randn(len(lens), hq, D, generator=g).to(torch.bfloat16)
    for i, (b, p) in enumerate(zip(batch_idx, pos)):
        rows = [(b, h, p, p + 1) for h in range(hq)]
        o, l = oracle.attend(_bits(q), out, indptr, indices, last, rows, hq=hq, hkv=hkv)
        for h in range(hq):
            np.testing.assert_array_equal(o[h], v_new[i, h // 2].double().numpy())
            s = float(q[b, h].double() @ k_new[i, h // 2].double()) / math.sqrt(D)
            assert abs(l[h] - s) < 1e-12


def test_out_of_range_tokens_skipped():
    indptr, indices, last, kv, g = _setup([5, 20], 16)
    k_new = torch.randn(4, 2, 16, generator=g).to(torch.bfloat16)
    out, skipped = oappend.append_kv(_bits(kv), _bits(k_new), _bits(k_new), [2, -1, 0, 1],
                                     [0, 0, 5, 19], indptr, indices, last, 16)
    assert skipped == [0, 1, 2]          # bad request, bad request, position == length
    changed = np.argwhere((out != _bits(kv)).any(axis=(-1, -2)))
    pages = {int(indices[indptr[1] + 19 // 16])}
    assert {int(c[0]) for c in changed} == pages


def test_hnd_read_back_through_attention_oracle():
    """HND cache: the appended rows read back through the attention oracle's
    HND gather, and the HND result is the NHD result with head and slot
    swapped."""
    lens, P, hkv, D = [23, 9, 40], 4, 2, 16
    indptr, indices, last, kv, g = _setup(lens, P, hkv=hkv, D=D, seed=5)
    kv_hnd = kv.permute(0, 1, 3, 2, 4).contiguous()
    batch_idx, pos = [0, 1, 2], [22, 3, 17]
    n = len(batch_idx)
    k_new = torch.randn(n, hkv, D, generator=g).to(torch.bfloat16)
    v_new = torch.randn(n, hkv, D, generator=g).to(torch.bfloat16)
    out_h, sk_h = oappend.append_kv(_bits(kv_hnd), _bits(k_new), _bits(v_new), batch_idx, pos,
                                    indptr, indices, last, P, layout="HND")
    out_n, sk_n = oappend.append_kv(_bits(kv), _bits(k_new), _bits(v_new), batch_idx, pos,
                                    indptr, indices, last, P)
    assert sk_h == sk_n == []
    for pg in range(out_n.shape[0]):
        for c in range(2):
            for s in range(P):
                for h in range(hkv):
                    assert np.array_equal(out_h[pg, c, h, s], out_n[pg, c, s, h])
    hq = 2 * hkv
    q = torch.randn(len(lens), hq, D, generator=g).to(torch.bfloat16)
    for i, (b, p) in enumerate(zip(batch_idx, pos)):
        rows = [(b, h, p, p + 1) for h in range(hq)]
        o, _ = oracle.attend(_bits(q), out_h, indptr, indices, last, rows, hq=hq, hkv=hkv,
                             layout="HND")
        for h in range(hq):
            np.testing.assert_array_equal(o[h], v_new[i, h // 2].double().numpy())
