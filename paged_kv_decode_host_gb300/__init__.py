"""Paged-KV GQA decode attention for GB300 -- thin Python binding of libpkd.

Every step of the computation runs in the CUDA library (``libpkd.so``, built
in-tree by :func:`build`); this module only marshals arguments: it checks
dtypes, shapes and devices, passes ``tensor.data_ptr()`` and the current
CUDA stream through ctypes (the per-step plan and run calls through the
small compiled ``_pkd_plan`` module when it was built), and raises on a non-zero
status.  There is no fallback: if the library is missing or was built for
another machine, loading it fails loudly.

API (names follow the pages' plan / run / merge_states):

* :class:`BatchDecodeWithPagedKVCache` -- ``plan(indptr, indices,
  last_page_len)`` (or ``plan_shared`` for a shared-prefix level) once per
  step, ``run(q, kv_cache)`` once per layer, ``capture(...)`` for a CUDA
  graph of a whole step.
* :func:`merge_states` -- exact LSE merge of two attention states.
* :func:`append_kv` -- write a step's new K / V rows into their page slots.
* :func:`plan_host` -- the scheduler alone on the host (no GPU), for tests.
* ``cascade=True`` contexts: ``plan_cascade(group_indptr, prefix, suffix)``
  plans a shared prefix and every request's own suffix together; ``run``
  returns attention over both, merged.
* :func:`selftest_bounded_wait` -- the device-side bounded-wait self-test.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

__all__ = [
    "build", "load", "PkdError", "BatchDecodeWithPagedKVCache", "merge_states", "append_kv",
    "append_kv_layers", "plan_host", "plan_host_shared", "plan_host_cascade", "advise_format",
    "schedule_layout",
    "selftest_bounded_wait", "Graph",
    "STATUS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkd.so")

STATUS = {
    0: "PKD_OK", -1: "PKD_E_INVALID_ARG", -2: "PKD_E_BAD_TABLE",
    -3: "PKD_E_UNSUPPORTED_SHAPE", -4: "PKD_E_WORKSPACE_TOO_SMALL",
    -5: "PKD_E_NO_PLAN", -6: "PKD_E_STALE_PLAN", -7: "PKD_E_CAPACITY",
    -8: "PKD_E_CUDA", -9: "PKD_E_DEVICE", -10: "PKD_E_SCRATCH_LIMIT",
}
DEV_ERR_TIMEOUT = 1
DEV_ERR_BOUNDS = 2
GRAPH_TIMING = 1

# Every entry point the C header declares (tests check the exports).
EXPORTS = (
    "pkd_workspace_bytes", "pkd_create", "pkd_destroy", "pkd_plan",
    "pkd_get_plan_info", "pkd_run", "pkd_merge_states", "pkd_last_device_error",
    "pkd_read_schedule", "pkd_plan_host", "pkd_schedule_layout",
    "pkd_graph_capture", "pkd_graph_capture_io", "pkd_graph_launch", "pkd_graph_layer_times",
    "pkd_graph_destroy", "pkd_status_str", "pkd_version", "pkd_run_static_scratch",
    "pkd_append_kv", "pkd_append_kv_ex", "pkd_plan_shared", "pkd_plan_host_shared", "pkd_run_scaled",
    "pkd_selftest_bounded_wait", "pkd_append_kv_layers", "pkd_static_scratch_last_error",
    "pkd_plan_cascade", "pkd_plan_host_cascade", "pkd_advise_format",
)


class PkdError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{what}: {self.name}" if what else self.name)


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_qo_heads", "num_kv_heads", "head_dim", "page_size", "max_batch",
        "max_num_pages", "num_pages", "alpha", "min_chunk_tokens", "num_ctas")] + [
        ("flags", ctypes.c_uint32)]


class FormatAdvice(ctypes.Structure):
    _fields_ = [("use_cascade", ctypes.c_int32), ("prefix_ctas", ctypes.c_int32),
                ("cascade_makespan", ctypes.c_int64), ("single_makespan", ctypes.c_int64),
                ("cascade_us", ctypes.c_float), ("single_us", ctypes.c_float)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class PlanInfo(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_ctas", ctypes.c_int32),
                ("chunk_tokens", ctypes.c_int32), ("num_items", ctypes.c_int32),
                ("num_units", ctypes.c_int32), ("num_slots", ctypes.c_int32),
                ("total_tokens", ctypes.c_int64), ("makespan", ctypes.c_int64),
                ("nnz", ctypes.c_int32), ("schedule_words", ctypes.c_int32),
                ("page_tiles", ctypes.c_int32), ("prefix_ctas", ctypes.c_int32),
                ("prefix_chunk_tokens", ctypes.c_int32)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


def build(force: bool = False) -> str:
    """Compile libpkd.so for sm_103a (in-tree)."""
    from . import _build
    return _build.build(force=force)


_lib = None


def load():
    """Load libpkd.so (must have been built with :func:`build`)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "paged_kv_decode_host_gb300.build() (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, u32, u64, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32,
                             ctypes.c_uint64, ctypes.c_size_t)
    cfgp = ctypes.POINTER(Config)
    sig = {
        "pkd_workspace_bytes": (sz, [cfgp]),
        "pkd_create": (ctypes.c_int, [cfgp, vp, sz, ctypes.POINTER(vp)]),
        "pkd_destroy": (None, [vp]),
        "pkd_plan": (ctypes.c_int, [vp, vp, vp, vp, i32, vp, ctypes.POINTER(u64)]),
        "pkd_get_plan_info": (ctypes.c_int, [vp, ctypes.POINTER(PlanInfo)]),
        "pkd_run": (ctypes.c_int, [vp, vp, vp, vp, vp, u64, vp]),
        "pkd_run_scaled": (ctypes.c_int, [vp, vp, vp, vp, vp, ctypes.c_float, ctypes.c_float,
                                          u64, vp]),
        "pkd_merge_states": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, i32, i32, i32, vp]),
        "pkd_last_device_error": (ctypes.c_int, [vp, vp, ctypes.POINTER(i32)]),
        "pkd_read_schedule": (ctypes.c_int, [vp, vp, sz, vp]),
        "pkd_plan_host": (ctypes.c_int, [cfgp, vp, vp, vp, i32, vp, sz,
                                         ctypes.POINTER(PlanInfo)]),
        "pkd_schedule_layout": (ctypes.c_int, [cfgp, vp]),
        "pkd_graph_capture": (ctypes.c_int, [vp, i32, vp, vp, vp, vp, vp, u32,
                                             ctypes.POINTER(vp)]),
        "pkd_graph_capture_io": (ctypes.c_int, [vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, u32,
                                                ctypes.POINTER(vp)]),
        "pkd_graph_launch": (ctypes.c_int, [vp, vp]),
        "pkd_graph_layer_times": (ctypes.c_int, [vp, vp]),
        "pkd_graph_destroy": (None, [vp]),
        "pkd_status_str": (ctypes.c_char_p, [ctypes.c_int]),
        "pkd_version": (ctypes.c_int, []),
        "pkd_run_static_scratch": (ctypes.c_int, [cfgp, vp, sz, vp, vp, vp, vp, vp]),
        "pkd_static_scratch_last_error": (ctypes.c_int, [cfgp, vp, ctypes.POINTER(i32)]),
        "pkd_plan_cascade": (ctypes.c_int, [vp, vp, i32, vp, vp, vp, vp, vp, vp, vp,
                                            ctypes.POINTER(u64)]),
        "pkd_plan_host_cascade": (ctypes.c_int, [cfgp, vp, i32, vp, vp, vp, vp, vp, vp, vp, sz,
                                                 ctypes.POINTER(PlanInfo)]),
        "pkd_advise_format": (ctypes.c_int, [cfgp, vp, i32, vp, vp, vp, vp,
                                             ctypes.POINTER(FormatAdvice)]),
        "pkd_append_kv": (ctypes.c_int, [vp, vp, vp, vp, i32, vp, vp, vp, i32, vp, i32, i32,
                                         i32, i32, vp, vp]),
        "pkd_append_kv_ex": (ctypes.c_int, [vp, vp, vp, vp, i32, vp, vp, vp, i32, vp, i32, i32,
                                            i32, i32, ctypes.c_uint32, vp, vp]),
        "pkd_plan_shared": (ctypes.c_int, [vp, vp, i32, vp, vp, vp, vp, ctypes.POINTER(u64)]),
        "pkd_plan_host_shared": (ctypes.c_int, [cfgp, vp, i32, vp, vp, vp, vp, sz,
                                                ctypes.POINTER(PlanInfo)]),
        "pkd_selftest_bounded_wait": (ctypes.c_int, [i32, vp, vp, vp]),
        "pkd_append_kv_layers": (ctypes.c_int, [i32, vp, vp, vp, vp, vp, i32, vp, vp, vp, i32,
                                                i32, i32, i32, i32, ctypes.c_uint32, vp, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _check(status, what):
    if status != 0:
        raise PkdError(status, what)


def _host_i32(a) -> np.ndarray:
    if type(a) is np.ndarray and a.dtype == np.int32 and a.flags.c_contiguous:
        return a   # the common case, checked first: plan() runs every decode step
    try:
        import torch
        if isinstance(a, torch.Tensor):
            if a.is_cuda:
                raise ValueError("page-table arrays are host arrays (the planner runs on the CPU)")
            if a.dtype != torch.int32:
                raise TypeError("page-table arrays must be int32")
            return np.ascontiguousarray(a.numpy())
    except ImportError:
        pass
    arr = np.asarray(a)
    if arr.dtype != np.int32:
        raise TypeError("page-table arrays must be int32 (int64 indices are rejected)")
    return np.ascontiguousarray(arr)


def _ptr(a: np.ndarray):
    return a.ctypes.data if a.size else None


FLAG_FMA_CONSUMER = 1   # fold the GQA group onto CUDA cores (fp32 FMA)
FLAG_MMA_CONSUMER = 2   # fold it onto tensor cores (mma.sync, bf16 in / fp32 acc)
FLAG_SHARED_PREFIX = 4  # shared-prefix context: plans over groups of requests
FLAG_KV_FP8 = 8         # E4M3 cache with per-call K / V scales
FLAG_ROW_COPIES = 16    # force one KV copy per token row (no page-tile tensor map)
FLAG_CHUNK_SEARCH = 64  # chunk = largest page multiple still giving >= N_CTA items
FLAG_HND = 32           # cache layout [pages, 2, Hkv, P, D] instead of NHD [pages, 2, P, Hkv, D]
FLAG_DENSE_PREFIX = 128  # shared prefix on tcgen05 tensor cores: 128-row tiles, one KV head per item
FLAG_CASCADE = 256      # both levels of a shared-prefix step in one plan, one launch, one merge


def make_config(num_qo_heads, num_kv_heads, head_dim, page_size, max_batch, max_num_pages,
                num_pages, alpha=-1, min_chunk_tokens=-1, num_ctas=0, flags=0) -> Config:
    return Config(num_qo_heads, num_kv_heads, head_dim, page_size, max_batch, max_num_pages,
                  num_pages, alpha, min_chunk_tokens, num_ctas, flags)


def schedule_layout(cfg: Config):
    lib = load()
    off = (ctypes.c_int64 * 6)()
    _check(lib.pkd_schedule_layout(ctypes.byref(cfg), off), "pkd_schedule_layout")
    return list(off)


def plan_host(cfg: Config, indptr, indices, last_page_len):
    """Run the C++ scheduler on the host.  Returns (words, info dict, layout)."""
    lib = load()
    indptr, indices, last = _host_i32(indptr), _host_i32(indices), _host_i32(last_page_len)
    off = schedule_layout(cfg)
    words = np.zeros(off[5], dtype=np.int32)
    info = PlanInfo()
    st = lib.pkd_plan_host(ctypes.byref(cfg), _ptr(indptr), _ptr(indices), _ptr(last),
                           int(last.shape[0]), _ptr(words), words.size, ctypes.byref(info))
    _check(st, "pkd_plan_host")
    return words, info.as_dict(), off


def plan_host_shared(cfg: Config, group_indptr, indptr, indices, last_page_len):
    """The C++ scheduler for a shared-prefix level, on the host."""
    lib = load()
    gi = _host_i32(group_indptr)
    indptr, indices, last = _host_i32(indptr), _host_i32(indices), _host_i32(last_page_len)
    off = schedule_layout(cfg)
    words = np.zeros(off[5], dtype=np.int32)
    info = PlanInfo()
    st = lib.pkd_plan_host_shared(ctypes.byref(cfg), _ptr(gi), int(last.shape[0]), _ptr(indptr),
                                  _ptr(indices), _ptr(last), _ptr(words), words.size,
                                  ctypes.byref(info))
    _check(st, "pkd_plan_host_shared")
    return words, info.as_dict(), off


def _cascade_tables(group_indptr, prefix, suffix):
    gi = _host_i32(group_indptr)
    p = [_host_i32(x) for x in prefix]
    q = [_host_i32(x) for x in suffix]
    n_groups = p[2].shape[0]
    batch = q[2].shape[0]
    if gi.shape[0] != n_groups + 1 or p[0].shape[0] != n_groups + 1:
        raise PkdError(-2, "group_indptr and the prefix indptr need one entry per group + 1")
    if q[0].shape[0] != batch + 1 or (n_groups and int(gi[-1]) != batch):
        raise PkdError(-2, "the suffix table needs one row per request of the groups")
    for ip, ix in ((p[0], p[1]), (q[0], q[1])):
        if ip.shape[0] > 1 and ix.shape[0] < ip[-1]:
            raise PkdError(-2, "indices shorter than indptr[-1]")
    return gi, n_groups, p, q


def plan_host_cascade(cfg: Config, group_indptr, prefix, suffix):
    """The C++ scheduler for a cascade step, on the host.  prefix = (indptr,
    indices, last_page_len) over groups, suffix = the same over requests."""
    lib = load()
    gi, n_groups, p, q = _cascade_tables(group_indptr, prefix, suffix)
    off = schedule_layout(cfg)
    words = np.zeros(off[5], dtype=np.int32)
    info = PlanInfo()
    st = lib.pkd_plan_host_cascade(ctypes.byref(cfg), _ptr(gi), n_groups, *[_ptr(x) for x in p],
                                   *[_ptr(x) for x in q], _ptr(words), words.size,
                                   ctypes.byref(info))
    _check(st, "pkd_plan_host_cascade")
    return words, info.as_dict(), off


def advise_format(cfg: Config, group_indptr, prefix, suffix):
    """Which format a shared-prefix step should take: the cascade plan or
    every request over its whole table (see pkd_advise_format).  cfg: a
    cascade configuration with num_ctas >= 2; prefix / suffix as for
    plan_cascade (page ids are not read).  Returns a dict with use_cascade
    and both predictions (microseconds per layer)."""
    lib = load()
    gi, n_groups, p, q = _cascade_tables(group_indptr, prefix, suffix)
    adv = FormatAdvice()
    _check(lib.pkd_advise_format(ctypes.byref(cfg), _ptr(gi), n_groups, _ptr(p[0]), _ptr(p[2]),
                                 _ptr(q[0]), _ptr(q[2]), ctypes.byref(adv)), "pkd_advise_format")
    return adv.as_dict()


def decode_schedule(words, off, info):
    """Unpack schedule words into python lists (same shape as the plan
    restatement's fields)."""
    n_cta, n_items, n_units, nnz = (info["num_ctas"], info["num_items"], info["num_units"],
                                    info["nnz"])
    cta_indptr = words[off[0]:off[0] + n_cta + 1].tolist()
    it = words[off[1]:off[1] + 8 * n_items].reshape(n_items, 8)
    items = [tuple(int(x) for x in r[:7]) for r in it]
    heads = [int(r[7]) for r in it]
    un = words[off[2]:off[2] + 2 * n_units].reshape(n_units, 2)
    units = [tuple(int(x) for x in r) for r in un]
    merge_indptr = words[off[3]:off[3] + n_units + 1].tolist()
    page_list = words[off[4]:off[4] + nnz].tolist()
    return dict(cta_indptr=cta_indptr, items=items, units=units, merge_indptr=merge_indptr,
                page_list=page_list, header=words[:32].tolist(), heads=heads)


_current_raw_stream = None
_fast_plan = None     # the CPython plan fast path (module), False when not built
_NOT_HANDLED = 1000   # its status for inputs it leaves to the general path


def _fast():
    """The compiled marshalling fast path for plan / plan_shared /
    plan_cascade / run, if built."""
    global _fast_plan
    if _fast_plan is None:
        try:
            from . import _pkd_plan as m
            lib = load()
            m.init(ctypes.cast(lib.pkd_plan, ctypes.c_void_p).value,
                   ctypes.cast(lib.pkd_plan_shared, ctypes.c_void_p).value,
                   ctypes.cast(lib.pkd_plan_cascade, ctypes.c_void_p).value,
                   ctypes.cast(lib.pkd_run_scaled, ctypes.c_void_p).value)
            _fast_plan = m
        except ImportError:
            _fast_plan = False
    return _fast_plan or None


def _stream_ptr(stream=None):
    """cudaStream_t of `stream`, else of torch's current stream on the
    current device (looked up without building a Stream object: plan / run
    are per-step host calls)."""
    global _current_raw_stream
    if stream is not None:
        return stream.cuda_stream
    if _current_raw_stream is None:
        import torch
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        dev = getattr(torch._C, "_cuda_getDevice", None)
        if raw is not None and dev is not None:
            _current_raw_stream = lambda: raw(dev())
        else:
            _current_raw_stream = lambda: torch.cuda.current_stream().cuda_stream
    return _current_raw_stream()


class Graph:
    """A captured decode step (``layers`` runs with fixed pointers)."""

    def __init__(self, owner, handle, layers, keep):
        self._owner = owner
        self._h = handle
        self.layers = layers
        self._keep = keep  # tensors whose addresses the graph holds

    def launch(self, stream=None):
        _check(load().pkd_graph_launch(self._h, _stream_ptr(stream)), "pkd_graph_launch")

    def layer_times(self):
        """Decode-kernel milliseconds of each layer in the last launch."""
        ms = (ctypes.c_float * self.layers)()
        _check(load().pkd_graph_layer_times(self._h, ms), "pkd_graph_layer_times")
        return list(ms)

    def close(self):
        if self._h:
            load().pkd_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class BatchDecodeWithPagedKVCache:
    """Plan once per decode step, run once per layer.

    The workspace is one device tensor allocated here with torch (its size
    and layout come from the library) and kept at a fixed address for the
    object's life.  q / out bf16; KV bf16 or e4m3, layout NHD
    ``[pages, 2, P, Hkv, D]`` or HND ``[pages, 2, Hkv, P, D]``.
    """

    def __init__(self, num_qo_heads, num_kv_heads, head_dim, page_size, *, max_batch,
                 max_num_pages, num_pages, alpha=-1, min_chunk_tokens=-1, num_ctas=0,
                 use_tensor_cores=None, shared_prefix=False, kv_dtype="bf16", kv_layout="NHD",
                 row_copies=False, chunk_rule="closed", dense_prefix=False, cascade=False,
                 device=None):
        import torch
        if kv_layout not in ("NHD", "HND"):
            raise ValueError("kv_layout must be 'NHD' [pages, 2, P, Hkv, D] or "
                             "'HND' [pages, 2, Hkv, P, D]")
        self.kv_layout = kv_layout
        lib = load()
        self.device = torch.device("cuda" if device is None else device)
        self.hq, self.hkv, self.d, self.p = num_qo_heads, num_kv_heads, head_dim, page_size
        self.num_pages = num_pages
        flags = 0 if use_tensor_cores is None else (
            FLAG_MMA_CONSUMER if use_tensor_cores else FLAG_FMA_CONSUMER)
        if shared_prefix:
            flags |= FLAG_SHARED_PREFIX
        if kv_dtype not in ("bf16", "e4m3"):
            raise ValueError("kv_dtype must be 'bf16' or 'e4m3'")
        self.kv_dtype = kv_dtype
        if kv_dtype == "e4m3":
            flags |= FLAG_KV_FP8
        if row_copies:
            flags |= FLAG_ROW_COPIES
        if kv_layout == "HND":
            flags |= FLAG_HND
        if dense_prefix:
            if not shared_prefix:
                raise ValueError("dense_prefix needs shared_prefix=True")
            flags |= FLAG_DENSE_PREFIX
        if cascade:
            if shared_prefix or dense_prefix or row_copies or kv_dtype != "bf16" or \
                    use_tensor_cores is False or chunk_rule != "closed":
                raise ValueError("a cascade context runs both levels itself: bf16 cache, "
                                 "tensor cores, the closed-form chunk rule")
            flags |= FLAG_CASCADE
        if chunk_rule not in ("closed", "search"):
            raise ValueError("chunk_rule must be 'closed' or 'search'")
        if chunk_rule == "search":
            flags |= FLAG_CHUNK_SEARCH
        self.cfg = make_config(num_qo_heads, num_kv_heads, head_dim, page_size, max_batch,
                               max_num_pages, num_pages, alpha, min_chunk_tokens, num_ctas, flags)
        with torch.cuda.device(self.device):
            nbytes = lib.pkd_workspace_bytes(ctypes.byref(self.cfg))
            if nbytes == 0:
                raise PkdError(-3, "pkd_workspace_bytes (invalid or unsupported configuration)")
            self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
            h = ctypes.c_void_p()
            _check(lib.pkd_create(ctypes.byref(self.cfg), ctypes.c_void_p(self.workspace.data_ptr()),
                                  nbytes, ctypes.byref(h)), "pkd_create")
        self._h = h
        self._hv = h.value
        self._lib = lib
        self._ep = ctypes.c_uint64()
        self._ep_ref = ctypes.byref(self._ep)
        self.epoch = 0
        self.batch = None
        self._run_shapes = None

    # -- plan ---------------------------------------------------------------
    def plan(self, indptr, indices, last_page_len, stream=None):
        """Schedule one decode step from host int32 arrays.  Returns the epoch."""
        fast = _fast()
        if fast is not None:
            st, ep = fast.plan(self._hv, indptr, indices, last_page_len, _stream_ptr(stream))
            if st != _NOT_HANDLED:
                if st:
                    _check(st, "pkd_plan")
                self.epoch = ep
                self.batch = len(last_page_len)
                return ep
        indptr, indices, last = _host_i32(indptr), _host_i32(indices), _host_i32(last_page_len)
        batch = last.shape[0]
        if indptr.shape[0] != batch + 1:
            raise PkdError(-2, "indptr must have batch + 1 entries")
        if batch and indices.shape[0] < indptr[batch]:
            raise PkdError(-2, "indices shorter than indptr[-1]")
        st = self._lib.pkd_plan(self._h, _ptr(indptr), _ptr(indices), _ptr(last), batch,
                                _stream_ptr(stream), self._ep_ref)
        if st:
            _check(st, "pkd_plan")
        self.epoch = self._ep.value
        self.batch = batch
        return self.epoch

    def plan_shared(self, group_indptr, indptr, indices, last_page_len, stream=None):
        """Plan a shared-prefix level: requests group_indptr[j] ..
        group_indptr[j+1]-1 attend over group j's pages (CSR over groups).
        Needs ``shared_prefix=True``.  Returns the epoch."""
        fast = _fast()
        if fast is not None:
            st, ep = fast.plan_shared(self._hv, group_indptr, indptr, indices, last_page_len,
                                      _stream_ptr(stream))
            if st != _NOT_HANDLED:
                if st:
                    _check(st, "pkd_plan_shared")
                self.epoch = ep
                self.batch = int(group_indptr[-1]) if len(last_page_len) else 0
                return ep
        gi = _host_i32(group_indptr)
        indptr, indices, last = _host_i32(indptr), _host_i32(indices), _host_i32(last_page_len)
        n_groups = last.shape[0]
        if gi.shape[0] != n_groups + 1 or indptr.shape[0] != n_groups + 1:
            raise PkdError(-2, "group_indptr and indptr need one entry per group + 1")
        st = self._lib.pkd_plan_shared(self._h, _ptr(gi), n_groups, _ptr(indptr), _ptr(indices),
                                       _ptr(last), _stream_ptr(stream), self._ep_ref)
        if st:
            _check(st, "pkd_plan_shared")
        self.epoch = self._ep.value
        self.batch = int(gi[-1]) if n_groups else 0
        return self.epoch

    def plan_cascade(self, group_indptr, prefix, suffix, stream=None):
        """Plan a cascade step (needs ``cascade=True``): requests
        group_indptr[j] .. group_indptr[j+1]-1 share group j's prefix pages,
        prefix = (indptr, indices, last_page_len) over groups; suffix = the
        same over requests, each request's own pages.  ``run`` then returns
        attention over prefix + suffix, merged.  Returns the epoch."""
        fast = _fast()
        if fast is not None:
            st, ep = fast.plan_cascade(self._hv, group_indptr, *prefix, *suffix,
                                       _stream_ptr(stream))
            if st != _NOT_HANDLED:
                if st:
                    _check(st, "pkd_plan_cascade")
                self.epoch = ep
                self.batch = len(suffix[2])
                return ep
        gi, n_groups, p, q = _cascade_tables(group_indptr, prefix, suffix)
        st = self._lib.pkd_plan_cascade(self._h, _ptr(gi), n_groups, *[_ptr(x) for x in p],
                                        *[_ptr(x) for x in q], _stream_ptr(stream),
                                        self._ep_ref)
        if st:
            _check(st, "pkd_plan_cascade")
        self.epoch = self._ep.value
        self.batch = int(q[2].shape[0])
        return self.epoch

    def plan_info(self):
        info = PlanInfo()
        _check(load().pkd_get_plan_info(self._h, ctypes.byref(info)), "pkd_get_plan_info")
        return info.as_dict()

    def schedule(self, stream=None):
        """The schedule words currently in the device workspace."""
        info = self.plan_info()
        off = schedule_layout(self._layout_cfg(info))
        words = np.zeros(off[4] + info["nnz"], dtype=np.int32)
        _check(load().pkd_read_schedule(self._h, _ptr(words), words.size, _stream_ptr(stream)),
               "pkd_read_schedule")
        return words, info, off

    def _layout_cfg(self, info):
        c = Config.from_buffer_copy(self.cfg)
        c.num_ctas = info["num_ctas"]
        return c

    # -- run ----------------------------------------------------------------
    def _check_run_args(self, q, kv_cache, out, lse):
        """Cheap checks of the common case (every attribute as planned); any
        mismatch goes to the full check, which names what is wrong."""
        import torch
        B = self.batch
        if B is not None:
            if self._run_shapes is None or self._run_shapes[0] != B:
                bf = torch.bfloat16
                self._run_shapes = (B, torch.Size((B, self.hq, self.d)),
                                    torch.Size((B, self.hq)),
                                    torch.Size((self.num_pages, 2, self.p, self.hkv, self.d)
                                               if self.kv_layout == "NHD" else
                                               (self.num_pages, 2, self.hkv, self.p, self.d)),
                                    bf, torch.bfloat16 if self.kv_dtype == "bf16"
                                    else torch.float8_e4m3fn, torch.float32,
                                    self.device.index)
            _, qs, ls, kvs, bf, kvd, f32, dev = self._run_shapes
            d = q.get_device()
            if (q.dtype is bf and out.dtype is bf and kv_cache.dtype is kvd
                    and q.shape == qs and out.shape == qs and kv_cache.shape == kvs
                    and q.is_contiguous() and out.is_contiguous() and kv_cache.is_contiguous()
                    and d >= 0 and (d == dev or dev is None) and out.get_device() == d
                    and kv_cache.get_device() == d
                    and (lse is None or (lse.dtype is f32 and lse.shape == ls
                                         and lse.is_contiguous()))):
                return
        self._check_run_args_full(q, kv_cache, out, lse)

    def _check_run_args_full(self, q, kv_cache, out, lse):
        import torch
        if self.batch is None:
            raise PkdError(-5, "run before plan")
        B = self.batch
        kv_dt = torch.bfloat16 if self.kv_dtype == "bf16" else torch.float8_e4m3fn
        for name, t, dt in (("q", q, torch.bfloat16), ("kv_cache", kv_cache, kv_dt),
                            ("out", out, torch.bfloat16)):
            if t.dtype != dt and not (name == "kv_cache" and self.kv_dtype == "e4m3"
                                      and t.dtype == torch.uint8):
                raise TypeError(f"{name} must be {dt} (planned kv_dtype "
                                f"{self.kv_dtype!r}), got {t.dtype}")
            if t.device != self.device and not (t.is_cuda and self.device.index is None):
                raise ValueError(f"{name} is on {t.device}, the plan on {self.device}")
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")
        if tuple(q.shape) != (B, self.hq, self.d):
            raise ValueError(f"q shape {tuple(q.shape)} != planned {(B, self.hq, self.d)}")
        if tuple(out.shape) != (B, self.hq, self.d):
            raise ValueError(f"out shape {tuple(out.shape)} != {(B, self.hq, self.d)}")
        want = ((self.num_pages, 2, self.p, self.hkv, self.d) if self.kv_layout == "NHD" else
                (self.num_pages, 2, self.hkv, self.p, self.d))
        if tuple(kv_cache.shape) != want:
            raise ValueError(f"kv_cache shape {tuple(kv_cache.shape)} is not "
                             f"{self.kv_layout} {want}")
        if lse is not None:
            if lse.dtype != torch.float32 or tuple(lse.shape) != (B, self.hq) or not lse.is_contiguous():
                raise ValueError("lse must be contiguous float32 [batch, Hq]")
        if (q.device != out.device or q.device != kv_cache.device
                or (lse is not None and lse.device != q.device)):
            raise ValueError("q, kv_cache, out and lse must be on one device")

    def run(self, q, kv_cache, out=None, lse=None, return_lse=True, expect_epoch=0,
            stream=None, k_scale=1.0, v_scale=1.0):
        """Attention for one layer.  Returns (out, lse) or out.  With scales
        the attended key is k_scale * K and the value v_scale * V (an E4M3
        cache needs them).  A nonzero expect_epoch (the value plan returned)
        also makes the kernels wait on the device for that plan's schedule,
        so the plan may run on another stream without an event."""
        import torch
        if out is None:
            out = torch.empty_like(q)
        if lse is None and return_lse:
            lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
        self._check_run_args(q, kv_cache, out, lse)
        fast = _fast()
        if fast is not None:
            st = fast.run(self._hv, q.data_ptr(), kv_cache.data_ptr(), out.data_ptr(),
                          lse.data_ptr() if lse is not None else 0, float(k_scale),
                          float(v_scale), int(expect_epoch), _stream_ptr(stream))
            if st != _NOT_HANDLED:
                _check(st, "pkd_run")
                return (out, lse) if return_lse else out
        st = load().pkd_run_scaled(self._h, ctypes.c_void_p(q.data_ptr()),
                                   ctypes.c_void_p(kv_cache.data_ptr()),
                                   ctypes.c_void_p(out.data_ptr()),
                                   ctypes.c_void_p(lse.data_ptr() if lse is not None else 0),
                                   float(k_scale), float(v_scale), int(expect_epoch),
                                   _stream_ptr(stream))
        _check(st, "pkd_run")
        return (out, lse) if return_lse else out

    def capture(self, qs, kvs, outs, lses=None, timing=False, kv_scales=None, host_qs=None,
                host_outs=None, host_lses=None) -> Graph:
        """Capture len(qs) runs (one decode step over all layers) in a graph.
        With host buffers (page-locked CPU tensors shaped like qs / outs /
        lses) the graph also copies each layer's queries in from host_qs and
        its results out to host_outs / host_lses, overlapped with the other
        layers' kernels."""
        import torch
        n = len(qs)
        for l in range(n):
            self._check_run_args(qs[l], kvs[l], outs[l], lses[l] if lses else None)
        for name, hs, ds in (("host_qs", host_qs, qs), ("host_outs", host_outs, outs),
                             ("host_lses", host_lses, lses)):
            if hs is None:
                continue
            if ds is None or len(hs) != n:
                raise ValueError(f"{name} needs one host tensor per layer (and the device side)")
            for h, d in zip(hs, ds):
                if (h.is_cuda or not h.is_pinned() or h.dtype != d.dtype or h.shape != d.shape
                        or not h.is_contiguous()):
                    raise ValueError(f"{name}: page-locked contiguous CPU tensors shaped and "
                                     f"typed like the device buffers")
        P = ctypes.c_void_p * n
        q_arr = P(*[t.data_ptr() for t in qs])
        kv_arr = P(*[t.data_ptr() for t in kvs])
        o_arr = P(*[t.data_ptr() for t in outs])
        l_arr = P(*[t.data_ptr() for t in lses]) if lses else None
        h = ctypes.c_void_p()
        as_vp = lambda a: ctypes.cast(a, ctypes.c_void_p) if a is not None else None
        sc = None
        if kv_scales is not None:
            sc = (ctypes.c_float * (2 * n))(*[float(x) for pair in kv_scales for x in pair])
        host = [P(*[t.data_ptr() for t in hs]) if hs is not None else None
                for hs in (host_qs, host_outs, host_lses)]
        st = load().pkd_graph_capture_io(self._h, n, as_vp(q_arr), as_vp(kv_arr), as_vp(o_arr),
                                         as_vp(l_arr), as_vp(sc), *[as_vp(a) for a in host],
                                         GRAPH_TIMING if timing else 0, ctypes.byref(h))
        _check(st, "pkd_graph_capture_io")
        return Graph(self, h, n, (list(qs), list(kvs), list(outs), list(lses or []), host_qs,
                                  host_outs, host_lses))

    def device_error(self, stream=None) -> int:
        v = ctypes.c_int32()
        _check(load().pkd_last_device_error(self._h, _stream_ptr(stream), ctypes.byref(v)),
               "pkd_last_device_error")
        return v.value

    def close(self):
        if getattr(self, "_h", None):
            load().pkd_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def selftest_bounded_wait(mode=0, device=None):
    """Run the device-side bounded-wait self-test (see pkd_selftest_bounded_wait)
    and wait for it.  Returns (error bits, [wait 0 ns, wait 1 ns])."""
    import torch
    dev = torch.device("cuda" if device is None else device)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ns = torch.zeros(2, dtype=torch.int64, device=dev)
    with torch.cuda.device(dev):
        _check(load().pkd_selftest_bounded_wait(int(mode), ctypes.c_void_p(err.data_ptr()),
                                                ctypes.c_void_p(ns.data_ptr()), _stream_ptr()),
               "pkd_selftest_bounded_wait")
        torch.cuda.synchronize(dev)
    return int(err.item()), [int(x) for x in ns.tolist()]


def merge_states(v_a, s_a, v_b, s_b, v_out=None, s_out=None, stream=None):
    """Exact merge of two attention states: v [n, H, D] bf16, s [n, H] fp32."""
    import torch
    for name, t, dt in (("v_a", v_a, torch.bfloat16), ("v_b", v_b, torch.bfloat16),
                        ("s_a", s_a, torch.float32), ("s_b", s_b, torch.float32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous CUDA {dt} tensor")
    if v_a.shape != v_b.shape or s_a.shape != s_b.shape or tuple(s_a.shape) != tuple(v_a.shape[:2]):
        raise ValueError("shape mismatch between the two states")
    if v_out is None:
        v_out = torch.empty_like(v_a)
    if s_out is None:
        s_out = torch.empty_like(s_a)
    n, H, D = v_a.shape
    st = load().pkd_merge_states(ctypes.c_void_p(v_a.data_ptr()), ctypes.c_void_p(s_a.data_ptr()),
                                 ctypes.c_void_p(v_b.data_ptr()), ctypes.c_void_p(s_b.data_ptr()),
                                 ctypes.c_void_p(v_out.data_ptr()),
                                 ctypes.c_void_p(s_out.data_ptr()), n, H, D, _stream_ptr(stream))
    _check(st, "pkd_merge_states")
    return v_out, s_out


def append_kv(k_new, v_new, batch_indices, positions, indptr, indices, last_page_len, kv_cache,
              err=None, stream=None, kv_layout="NHD"):
    """append_paged_kv_cache: write new tokens' K / V rows into their page slots.

    k_new, v_new: [n, Hkv, D], the cache's dtype (bf16, or e4m3 bytes);
    batch_indices, positions: int32 [n] (position = 0-based index of the
    token in its request after the append); indptr / indices / last_page_len:
    int32 CUDA tensors, the table after the append; kv_cache: NHD
    [pages, 2, P, Hkv, D] or HND [pages, 2, Hkv, P, D], written in place.
    err: optional int32 CUDA tensor of one element; tokens outside the table
    are skipped and flagged there."""
    import torch
    fp8 = kv_cache.dtype in (torch.float8_e4m3fn, torch.uint8)
    kv_dt = kv_cache.dtype if fp8 else torch.bfloat16
    for name, t, dt in (("k_new", k_new, kv_dt), ("v_new", v_new, kv_dt),
                        ("kv_cache", kv_cache, kv_dt),
                        ("batch_indices", batch_indices, torch.int32),
                        ("positions", positions, torch.int32), ("indptr", indptr, torch.int32),
                        ("indices", indices, torch.int32),
                        ("last_page_len", last_page_len, torch.int32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous CUDA {dt} tensor")
    if kv_layout not in ("NHD", "HND"):
        raise ValueError("kv_layout must be 'NHD' or 'HND'")
    n = int(k_new.shape[0])
    if kv_layout == "NHD":
        pages, two, P, hkv, D = kv_cache.shape
    else:
        pages, two, hkv, P, D = kv_cache.shape
    if two != 2 or tuple(k_new.shape) != (n, hkv, D) or v_new.shape != k_new.shape:
        raise ValueError(f"k_new / v_new must be [n, Hkv, D] matching the {kv_layout} cache")
    if batch_indices.numel() != n or positions.numel() != n:
        raise ValueError("batch_indices and positions need one entry per new token")
    batch = int(last_page_len.numel())
    if indptr.numel() != batch + 1:
        raise ValueError("indptr must have batch + 1 entries")
    if err is not None and (err.dtype != torch.int32 or not err.is_cuda):
        raise TypeError("err must be an int32 CUDA tensor")
    flags = (FLAG_HND if kv_layout == "HND" else 0) | (FLAG_KV_FP8 if fp8 else 0)
    st = load().pkd_append_kv_ex(
        ctypes.c_void_p(k_new.data_ptr()), ctypes.c_void_p(v_new.data_ptr()),
        ctypes.c_void_p(batch_indices.data_ptr()), ctypes.c_void_p(positions.data_ptr()), n,
        ctypes.c_void_p(indptr.data_ptr()), ctypes.c_void_p(indices.data_ptr()),
        ctypes.c_void_p(last_page_len.data_ptr()), batch, ctypes.c_void_p(kv_cache.data_ptr()),
        int(pages), int(P), int(hkv), int(D), flags,
        ctypes.c_void_p(err.data_ptr() if err is not None else 0), _stream_ptr(stream))
    _check(st, "pkd_append_kv_ex")
    return kv_cache


def append_kv_layers(k_news, v_news, batch_indices, positions, indptr, indices, last_page_len,
                     kv_caches, err=None, stream=None, kv_layout="NHD"):
    """append_kv for every layer of a step in one launch: layer l's rows
    k_news[l] / v_news[l] go into kv_caches[l]; the layers share the tokens
    and the page table (arguments otherwise as append_kv)."""
    import torch
    layers = len(kv_caches)
    if not 1 <= layers <= 128 or len(k_news) != layers or len(v_news) != layers:
        raise ValueError("one k_new, v_new and cache per layer, 1 to 128 layers")
    c0, k0 = kv_caches[0], k_news[0]
    for l in range(layers):
        for name, t, ref in (("kv_caches", kv_caches[l], c0), ("k_news", k_news[l], k0),
                             ("v_news", v_news[l], k0)):
            if t.dtype != ref.dtype or t.shape != ref.shape or not t.is_cuda or \
                    not t.is_contiguous():
                raise ValueError(f"{name}[{l}] must match layer 0's dtype and shape "
                                 "(contiguous, on the GPU)")
    fp8 = c0.dtype in (torch.float8_e4m3fn, torch.uint8)
    kv_dt = c0.dtype if fp8 else torch.bfloat16
    for name, t, dt in (("k_new", k0, kv_dt), ("kv_cache", c0, kv_dt),
                        ("batch_indices", batch_indices, torch.int32),
                        ("positions", positions, torch.int32), ("indptr", indptr, torch.int32),
                        ("indices", indices, torch.int32),
                        ("last_page_len", last_page_len, torch.int32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous CUDA {dt} tensor")
    if kv_layout not in ("NHD", "HND"):
        raise ValueError("kv_layout must be 'NHD' or 'HND'")
    n = int(k0.shape[0])
    if kv_layout == "NHD":
        pages, two, P, hkv, D = c0.shape
    else:
        pages, two, hkv, P, D = c0.shape
    if two != 2 or tuple(k0.shape) != (n, hkv, D):
        raise ValueError(f"k_new / v_new must be [n, Hkv, D] matching the {kv_layout} cache")
    if batch_indices.numel() != n or positions.numel() != n:
        raise ValueError("batch_indices and positions need one entry per new token")
    batch = int(last_page_len.numel())
    if indptr.numel() != batch + 1:
        raise ValueError("indptr must have batch + 1 entries")
    if err is not None and (err.dtype != torch.int32 or not err.is_cuda):
        raise TypeError("err must be an int32 CUDA tensor")
    flags = (FLAG_HND if kv_layout == "HND" else 0) | (FLAG_KV_FP8 if fp8 else 0)

    def ptrs(ts):
        return (ctypes.c_void_p * layers)(*[t.data_ptr() for t in ts])

    st = load().pkd_append_kv_layers(
        layers, ptrs(k_news), ptrs(v_news), ptrs(kv_caches),
        ctypes.c_void_p(batch_indices.data_ptr()), ctypes.c_void_p(positions.data_ptr()), n,
        ctypes.c_void_p(indptr.data_ptr()), ctypes.c_void_p(indices.data_ptr()),
        ctypes.c_void_p(last_page_len.data_ptr()), batch, int(pages), int(P), int(hkv), int(D),
        flags, ctypes.c_void_p(err.data_ptr() if err is not None else 0), _stream_ptr(stream))
    _check(st, "pkd_append_kv_layers")
    return kv_caches
