"""GPU parity of append_paged_kv_cache against the numpy oracle: the whole
cache must match bit for bit (a copy), tokens outside the table are skipped
and flagged, never written."""
import numpy as np
import pytest
import torch

import paged_kv_decode_host_gb300 as pkd
import workloads
from oracle import append as oappend

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkd.build()
    pkd.load()


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("P,hkv,D", [(16, 8, 128), (1, 8, 128), (3, 4, 64), (32, 2, 128)])
def test_append_matches_oracle(P, hkv, D):
    rng = np.random.default_rng(P * 7 + hkv)
    lens = rng.integers(1, 300, 24).tolist()
    pool = sum(-(-l // P) for l in lens) + 9
    ids = rng.permutation(pool).astype(np.int32)
    indptr, indices, last = workloads.page_table(lens, P, ids)
    g = torch.Generator(device="cuda").manual_seed(5)
    kv = torch.randn(pool, 2, P, hkv, D, generator=g, device="cuda").to(torch.bfloat16)
    # one decode token per request (its last position) plus random positions
    b = list(range(len(lens))) + rng.integers(0, len(lens), 40).tolist()
    pos = [lens[i] - 1 for i in range(len(lens))] + [int(rng.integers(0, lens[i])) for i in b[len(lens):]]
    # bad entries: unknown request, negative position, position == length
    b += [len(lens) + 3, 0, 5]
    pos += [0, -1, lens[5]]
    # distinct targets so the result does not depend on write order
    seen, keep = set(), []
    for i, (bb, pp) in enumerate(zip(b, pos)):
        key = (bb, pp)
        if key not in seen:
            seen.add(key)
            keep.append(i)
    b = [b[i] for i in keep]
    pos = [pos[i] for i in keep]
    n = len(b)
    k_new = torch.randn(n, hkv, D, generator=g, device="cuda").to(torch.bfloat16)
    v_new = torch.randn(n, hkv, D, generator=g, device="cuda").to(torch.bfloat16)
    ref, skipped = oappend.append_kv(_bits(kv), _bits(k_new), _bits(v_new), b, pos,
                                     indptr, indices, last, P)
    assert len(skipped) == 3
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = lambda a: torch.tensor(np.asarray(a, dtype=np.int32), device="cuda")
    pkd.append_kv(k_new, v_new, dev(b), dev(pos), dev(indptr), dev(indices), dev(last), kv,
                  err=err)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_bits(kv), ref)
    assert int(err.item()) == pkd.DEV_ERR_BOUNDS


def test_append_then_decode_reads_new_token():
    """Append the step's token, then decode: the attention over a request
    whose only token was just appended returns that token's V row."""
    P, hq, hkv, D = 16, 32, 8, 128
    lens = [1, 1]
    indptr, indices, last = workloads.page_table(lens, P, np.array([3, 1], np.int32))
    kv = torch.zeros(5, 2, P, hkv, D, dtype=torch.bfloat16, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(2)
    k_new = torch.randn(2, hkv, D, generator=g, device="cuda").to(torch.bfloat16)
    v_new = torch.randn(2, hkv, D, generator=g, device="cuda").to(torch.bfloat16)
    dev = lambda a: torch.tensor(np.asarray(a, dtype=np.int32), device="cuda")
    pkd.append_kv(k_new, v_new, dev([0, 1]), dev([0, 0]), dev(indptr), dev(indices), dev(last), kv)
    dec = pkd.BatchDecodeWithPagedKVCache(hq, hkv, D, P, max_batch=2, max_num_pages=2,
                                          num_pages=5)
    dec.plan(indptr, indices, last)
    q = torch.randn(2, hq, D, generator=g, device="cuda").to(torch.bfloat16)
    out, lse = dec.run(q, kv)
    torch.cuda.synchronize()
    for i in range(2):
        for h in range(hq):
            assert torch.equal(out[i, h], v_new[i, h // (hq // hkv)])


@pytest.mark.parametrize("layout,fp8", [("NHD", False), ("HND", False), ("NHD", True)])
def test_append_layers_matches_oracle_per_layer(layout, fp8):
    """pkd_append_kv_layers: one launch writes every layer's rows; each
    layer's cache equals the oracle's append of that layer's rows, bit for
    bit, and tokens outside the table are skipped in every layer."""
    P, hkv, D, layers = 16, 8, 128, 5
    rng = np.random.default_rng(91 + 2 * fp8 + (layout == "HND"))
    lens = rng.integers(1, 200, 12).tolist()
    pool = sum(-(-l // P) for l in lens) + 5
    indptr, indices, last = workloads.page_table(lens, P, rng.permutation(pool).astype(np.int32))
    b = list(range(len(lens))) + [len(lens) + 2]          # the last one is outside the table
    pos = [l - 1 for l in lens] + [0]
    n = len(b)
    g = torch.Generator(device="cuda").manual_seed(13)
    shape = (pool, 2, P, hkv, D) if layout == "NHD" else (pool, 2, hkv, P, D)

    def rnd(*s):
        x = torch.randn(*s, generator=g, device="cuda")
        return x.to(torch.float8_e4m3fn) if fp8 else x.to(torch.bfloat16)

    kvs = [rnd(*shape) for _ in range(layers)]
    ks = [rnd(n, hkv, D) for _ in range(layers)]
    vs = [rnd(n, hkv, D) for _ in range(layers)]
    bits = (lambda t: t.detach().cpu().contiguous().view(torch.uint8).numpy()) if fp8 else _bits
    refs = []
    for l in range(layers):
        ref, skipped = oappend.append_kv(bits(kvs[l]), bits(ks[l]), bits(vs[l]), b, pos,
                                         indptr, indices, last, P, layout=layout)
        assert len(skipped) == 1
        refs.append(ref)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = lambda a: torch.tensor(np.asarray(a, dtype=np.int32), device="cuda")
    pkd.append_kv_layers(ks, vs, dev(b), dev(pos), dev(indptr), dev(indices), dev(last), kvs,
                         err=err, kv_layout=layout)
    torch.cuda.synchronize()
    for l in range(layers):
        np.testing.assert_array_equal(bits(kvs[l]), refs[l])
    assert int(err.item()) == pkd.DEV_ERR_BOUNDS


def test_append_layers_rejects_bad_arguments():
    kv = torch.zeros(4, 2, 16, 8, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 8, 128, dtype=torch.bfloat16, device="cuda")
    i32 = torch.zeros(1, dtype=torch.int32, device="cuda")
    ip = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):                       # no layers
        pkd.append_kv_layers([], [], i32, i32, ip, i32, i32, [])
    with pytest.raises(ValueError):                       # layer shapes differ
        pkd.append_kv_layers([k, k], [k, k], i32, i32, ip, i32, i32, [kv, kv[:2].clone()])
    lib = pkd.load()
    assert lib.pkd_append_kv_layers(0, None, None, None, None, None, 1, None, None, None, 1, 4,
                                    16, 8, 128, 0, None, None) == -1
