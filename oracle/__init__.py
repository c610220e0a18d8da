"""CPU reference oracle for paged-KV decode attention -- TEST INFRASTRUCTURE.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this package.  The CUDA library never links, loads or calls it,
and it never calls the CUDA library: the two share no code.

* ``oracle.c``  -- fp64 attention, attention states and their merge (C,
  pthreads), built by :func:`build` with the host C compiler.
* ``plan.py``   -- a plain-Python restatement of the host scheduler.

Every function here cites, in ``oracle.c`` / ``plan.py``, the passage of the
pages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import plan  # noqa: F401  (re-export)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

OK, E_ARG, E_TABLE, E_SELFCHECK = 0, -1, -2, -3


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
               "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        p = ctypes.c_void_p
        i = ctypes.c_int
        lib.oracle_lengths.argtypes = [p, p, p, i, i, i, p]
        lib.oracle_attend.argtypes = [p, p, p, p, p, i, i, i, i, i, i, p, i, p, p, i]
        lib.oracle_merge.argtypes = [p, p, p, p, i, i, p, p]
        d = ctypes.c_double
        lib.oracle_attend_ex.argtypes = [p, p, i, i, d, d, p, p, p, i, i, i, i, i, i, p, i, p,
                                         p, i]
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_double.restype = d
        for f in (lib.oracle_lengths, lib.oracle_attend, lib.oracle_merge, lib.oracle_attend_ex):
            f.restype = i
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits(t) -> np.ndarray:
    """bf16 torch tensor -> contiguous uint16 numpy array of its bit patterns."""
    import torch
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def lengths(indptr, indices, last, page_size: int, num_pages: int) -> np.ndarray:
    """Per-request KV lengths l = P (n - 1) + r after the table check."""
    lib = _load()
    indptr, indices, last = _i32(indptr), _i32(indices), _i32(last)
    batch = last.shape[0]
    out = np.zeros(max(batch, 1), dtype=np.int64)
    st = lib.oracle_lengths(_ptr(indptr), _ptr(indices), _ptr(last), batch,
                            page_size, num_pages, _ptr(out))
    if st != OK:
        raise OracleError(f"oracle_lengths: status {st}")
    return out[:batch]


_LAYOUTS = {"NHD": 0, "HND": 1}


def _rows4(rows):
    rows = np.asarray(rows, dtype=np.int32)
    if rows.ndim == 1:
        rows = rows.reshape(-1, 2)
    if rows.shape[1] == 2:
        rows = np.concatenate([rows, np.zeros((rows.shape[0], 1), np.int32),
                               -np.ones((rows.shape[0], 1), np.int32)], axis=1)
    return np.ascontiguousarray(rows)


def _cache_dims(shape, layout):
    """(pages, P, Hkv, D) of a cache shape in the given layout."""
    if layout == "NHD":
        pages, two, P, hkv, D = shape
    elif layout == "HND":
        pages, two, hkv, P, D = shape
    else:
        raise ValueError("layout must be 'NHD' or 'HND'")
    assert two == 2
    return pages, P, hkv, D


def _attend(qb, kvb, kv_type, layout, k_scale, v_scale, indptr, indices, last, rows, hq, hkv,
            nthreads):
    lib = _load()
    B, hq_, D = qb.shape
    pages, P, hkv_, D2 = _cache_dims(kvb.shape, layout)
    assert hq_ == hq and hkv_ == hkv and D2 == D
    rows = _rows4(rows)
    n = rows.shape[0]
    out = np.zeros((max(n, 1), D), dtype=np.float64)
    lse = np.zeros(max(n, 1), dtype=np.float64)
    indptr, indices, last = _i32(indptr), _i32(indices), _i32(last)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    st = lib.oracle_attend_ex(_ptr(qb), _ptr(kvb), kv_type, _LAYOUTS[layout], float(k_scale),
                              float(v_scale), _ptr(indptr), _ptr(indices), _ptr(last), B, hq,
                              hkv, D, P, pages, _ptr(rows), n, _ptr(out), _ptr(lse),
                              int(nthreads))
    if st != OK:
        raise OracleError(f"oracle_attend_ex: status {st}")
    return out[:n], lse[:n]


def attend(q, kv, indptr, indices, last, rows, *, hq: int, hkv: int,
           nthreads: int | None = None, layout: str = "NHD"):
    """Attention states for query rows.

    q: bf16 [B, Hq, D]; kv: bf16 [pages, 2, P, Hkv, D] (NHD) or
    [pages, 2, Hkv, P, D] (HND).
    rows: int array (n, 2) of (request, query head) -- the full KV range -- or
    (n, 4) of (request, query head, t0, t1) for the partial state of tokens
    [t0, t1).  Returns (out [n, D] float64, lse [n] float64, natural log).
    """
    return _attend(_bits(q), _bits(kv), 0, layout, 1.0, 1.0, indptr, indices, last, rows, hq,
                   hkv, nthreads)


def e4m3_to_float(byte: int) -> float:
    """Decode one E4M3 byte (the oracle's own decoder)."""
    return float(_load().oracle_e4m3_to_double(int(byte)))


def _u8(t) -> np.ndarray:
    """E4M3 cache (torch float8_e4m3fn / uint8 tensor or numpy uint8) -> uint8 numpy."""
    import torch
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint8
        return np.ascontiguousarray(t)
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def attend_fp8(q, kv8, indptr, indices, last, rows, *, hq: int, hkv: int, k_scale: float,
               v_scale: float, nthreads: int | None = None, layout: str = "NHD"):
    """attend() for an E4M3 cache with K / V scales (bytes, NHD or HND)."""
    return _attend(_bits(q), _u8(kv8), 1, layout, k_scale, v_scale, indptr, indices, last, rows,
                   hq, hkv, nthreads)


def decode_fp8(q, kv8, indptr, indices, last, *, hq: int, hkv: int, k_scale: float,
               v_scale: float, nthreads=None, layout: str = "NHD"):
    """Full decode attention over an E4M3 cache: out [B, Hq, D], lse [B, Hq]."""
    B = int(np.asarray(last).shape[0])
    rows = np.array([(i, h) for i in range(B) for h in range(hq)], dtype=np.int32)
    out, lse = attend_fp8(q, kv8, indptr, indices, last, rows.reshape(-1, 2), hq=hq, hkv=hkv,
                          k_scale=k_scale, v_scale=v_scale, nthreads=nthreads, layout=layout)
    return out.reshape(B, hq, -1), lse.reshape(B, hq)


def decode(q, kv, indptr, indices, last, *, hq: int, hkv: int, nthreads=None,
           layout: str = "NHD"):
    """Full decode attention: out [B, Hq, D] and lse [B, Hq] (float64)."""
    B = int(np.asarray(last).shape[0])
    rows = np.array([(i, h) for i in range(B) for h in range(hq)], dtype=np.int32)
    out, lse = attend(q, kv, indptr, indices, last, rows.reshape(-1, 2),
                      hq=hq, hkv=hkv, nthreads=nthreads, layout=layout)
    D = out.shape[1] if out.size else (_bits(q).shape[2])
    return out.reshape(B, hq, D), lse.reshape(B, hq)


def merge(o_a, l_a, o_b, l_b):
    """Merge two attention states elementwise; shapes o [..., D], l [...]."""
    lib = _load()
    o_a = np.ascontiguousarray(o_a, dtype=np.float64)
    o_b = np.ascontiguousarray(o_b, dtype=np.float64)
    l_a = np.ascontiguousarray(l_a, dtype=np.float64)
    l_b = np.ascontiguousarray(l_b, dtype=np.float64)
    D = o_a.shape[-1]
    n = int(np.prod(l_a.shape)) if l_a.ndim else 1
    o = np.zeros_like(o_a)
    l = np.zeros_like(l_a)
    lib.oracle_merge(_ptr(o_a), _ptr(l_a), _ptr(o_b), _ptr(l_b), n, D, _ptr(o), _ptr(l))
    return o, l
