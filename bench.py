"""Decode-step benchmark: achieved HBM GB/s (and % of peak) and steps/s.

Default workload: the Llama-3-8B-shaped decode step -- 32 layers, Hq 32,
Hkv 8, D 128, bf16, page size 16, 64 requests with KV lengths uniform in
[1, 8192] (seeded), pages scattered over the pool.  One step = plan on the
host (schedule copied into the fixed workspace) + one CUDA-graph replay of
the 32 per-layer runs (decode kernel + split merge each).

Throughput counts ALGORITHMIC bytes: the valid K and V rows of every request
(sum_i l_i x 2 x Hkv x D x 2 per layer), q, out, lse and the page table --
not partials, unused slots of last pages or the schedule.  Per-layer caches
(1.17 GB each) are larger than L2, and consecutive layers read different
caches, so no flush is needed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llama8b_step|skewed|token_sparse|shared_prefix]

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle on a bounded sample of the same workload (the reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "decode-step KV throughput: achieved HBM GB/s (% of GB300 peak) and steps/s"
FALLBACK_HBM_GBS = 6800.0
PROFILE_DIR = os.path.join(ROOT, "profiles")
# the decode kernel's sources: a profile's counters stand for the kernel built from these
KERNEL_SOURCES = [os.path.join(ROOT, "paged_kv_decode_host_gb300", "csrc", f)
                  for f in ("decode_kernel.cu", "sm103_ptx.cuh", "pkd_internal.h",
                            "prefix_tc_body.cuh")]


def kernel_source_sha256():
    h = hashlib.sha256()
    for path in KERNEL_SOURCES:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# --------------------------------------------------------------------- bytes

def alg_bytes_per_layer(w, lens, nnz):
    kv = sum(lens) * 2 * w.hkv * w.head_dim * w.kv_elem_bytes
    q = w.batch * w.hq * w.head_dim * 2
    out = w.batch * w.hq * w.head_dim * 2
    lse = w.batch * w.hq * 4
    table = 4 * (nnz + 2 * w.batch + 1)
    return kv + q + out + lse + table


def _lens(t, P):
    ip, last = t["indptr"], t["last"]
    return [int(P * (ip[i + 1] - ip[i] - 1) + last[i]) for i in range(len(last))]


# -------------------------------------------------------------------- peaks

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def traffic_from_profile(workload, kernel="decode_kernel"):
    """DRAM bytes per launch of this workload's dominant kernel from the
    committed ncu summary (profiles/<kernel>_<workload>.md), if it was taken
    on the current kernel source (else None)."""
    try:
        with open(os.path.join(PROFILE_DIR, f"{kernel}_{workload}.md")) as f:
            text = f.read()
        sha = kernel_source_sha256()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256") != sha:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id, period_ms=20):
        self.gpu_id = gpu_id
        self.period_ms = period_ms   # query-only sampling; short timed regions need a fast rate
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_id), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- multi-rank

def max_over_ranks(ms, world, device):
    """Whole-job time = the slowest rank's (replicas run independent shards,
    no data-path collective; this is the only exchange, timing metadata)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    tt = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def aggregate_throughput(bytes_per_rank_step, ms_per_step, world):
    """GB/s of the whole job: every rank moved bytes_per_rank_step per step,
    in the slowest rank's time."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


# ---------------------------------------------------------------- our arm

def _views(w, t, prefix_mode="cascade"):
    """(name, group_indptr or None, tables) per planned context.  The shared
    prefix is one group: every request over the prefix pages (FlashInfer
    完全拆解, Composable Format).  "cascade": one context plans the prefix
    level and the suffixes together (tables = (prefix, suffix)); "levels":
    a shared-prefix context and a plain one, joined by merge_states."""
    if w.prefix_tokens:
        n_pre = w.prefix_tokens // w.page_size
        prefix = (np.array([0, n_pre], np.int32), np.asarray(t["prefix"][1][:n_pre], np.int32),
                  np.array([w.page_size], np.int32))
        gi = np.array([0, w.batch], np.int32)
        if prefix_mode == "cascade":
            return [("cascade", gi, (prefix, t["suffix"]))]
        return [("prefix", gi, prefix), ("suffix", None, t["suffix"])]
    return [("full", None, (t["indptr"], t["indices"], t["last"]))]


def _nnz(name, table):
    if name == "cascade":
        return int(table[0][0][-1]) + int(table[1][0][-1])
    return int(table[0][-1])


def _plan(d, group_indptr, table, stream=None, name=None):
    if name == "cascade":
        d.plan_cascade(group_indptr, table[0], table[1], stream=stream)
    elif group_indptr is None:
        d.plan(*table, stream=stream)
    else:
        d.plan_shared(group_indptr, *table, stream=stream)


class _ComposedGraph:
    """A torch CUDA graph of one shared-prefix step: the prefix level and the
    suffix level (each a decode + merge through the C ABI) on two streams,
    joined by merge_states."""

    layers = 1

    def __init__(self, g):
        self.g = g

    def launch(self):
        self.g.replay()

    def close(self):
        self.g = None


def _composed_step_graph(ds, q, kv, po, pl, so, sl, out, lse, side, dev, io=None):
    """io = (copy streams (in, out), [(device dst, host src)], [(host dst,
    device src)]): copies captured on two branches of the graph that run
    beside the step's kernels (the next step's q in, the previous step's
    results out)."""
    import torch

    import paged_kv_decode_host_gb300 as pkd
    main = torch.cuda.Stream(device=dev)
    # warm up outside the capture (plans are already published)
    with torch.cuda.stream(main):
        ds[0].run(q, kv, out=po, lse=pl)
        ds[1].run(q, kv, out=so, lse=sl)
        pkd.merge_states(po, pl, so, sl, out, lse)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=main):
        fork = torch.cuda.Event()
        fork.record(main)
        side.wait_event(fork)
        if io is not None:
            (s_in, s_out), copies_in, copies_out = io
            for st, pairs in ((s_in, copies_in), (s_out, copies_out)):
                st.wait_event(fork)
                with torch.cuda.stream(st):
                    for dst, src in pairs:
                        dst.copy_(src, non_blocking=True)
        ds[0].run(q, kv, out=po, lse=pl)
        with torch.cuda.stream(side):
            ds[1].run(q, kv, out=so, lse=sl)
        main.wait_stream(side)
        pkd.merge_states(po, pl, so, sl, out, lse)
        if io is not None:
            main.wait_stream(s_in)
            main.wait_stream(s_out)
    return _ComposedGraph(g)


def _cascade_step_graph(dec, q, kv, out, lse, dev, io):
    """A torch CUDA graph of one cascade step (the launch and its merge)
    with, on two branches beside it, the next step's q copied in from pinned
    host memory and the previous step's out + lse copied back (io = ((in
    stream, out stream), [(device dst, host src)], [(host dst, device
    src)]))."""
    import torch
    main = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(main):
        dec.run(q, kv, out=out, lse=lse)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    (s_in, s_out), copies_in, copies_out = io
    with torch.cuda.graph(g, stream=main):
        fork = torch.cuda.Event()
        fork.record(main)
        for st, pairs in ((s_in, copies_in), (s_out, copies_out)):
            st.wait_event(fork)
            with torch.cuda.stream(st):
                for dst, src in pairs:
                    dst.copy_(src, non_blocking=True)
        dec.run(q, kv, out=out, lse=lse)
        main.wait_stream(s_in)
        main.wait_stream(s_out)
    return _ComposedGraph(g)


def run_ours(args, rank, world):
    import torch

    import paged_kv_decode_host_gb300 as pkd

    pkd.build()
    pkd.load()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = workloads.workload(args.workload)
    t = workloads.make_tables(w)
    P = w.page_size
    lens = _lens(t, P)
    nnz = int(t["indptr"][-1])
    layers = args.layers if args.layers > 0 else w.layers
    # distinct caches per replay for single-layer workloads so no step reads
    # another step's bytes out of L2: at least 4, and enough that the other
    # copies read between two reads of one copy hold twice the L2.  No more:
    # each copy is one more graph in the rotation, and replaying N distinct
    # graphs in turn costs about 0.1 us per launch per graph.
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    pool_bytes = w.pool_pages * 2 * P * w.hkv * w.head_dim * w.kv_elem_bytes
    copies = 1 if layers > 1 else max(4, 1 + int(np.ceil(2 * l2 / pool_bytes)))
    if args.copies > 0:   # fewer cache copies (a smaller device footprint for counter captures)
        copies = args.copies
    n_kv = layers * copies
    if w.kv_dtype == "e4m3":
        kvs, kv_scale = workloads.make_kv_fp8(w, device=dev, layers=n_kv)
        kv_scales = [(kv_scale, kv_scale)] * layers
    else:
        kvs = workloads.make_kv(w, device=dev, layers=n_kv)
        kv_scales = None
    qs = workloads.make_q(w, device=dev, layers=layers)
    outs = [torch.empty_like(x) for x in qs]
    lses = [torch.empty(w.batch, w.hq, dtype=torch.float32, device=dev) for _ in qs]
    views = _views(w, t, args.prefix_mode)
    cascade = views[0][0] == "cascade"
    # Two planning contexts used on alternate steps: the schedule of step k+1
    # is uploaded on a copy stream while step k's kernels run (each context's
    # workspace is rewritten only after the step that last read it is done).
    n_sets = 2
    sets = []
    for _ in range(n_sets):
        decs = []
        for name, gi, tables in views:
            d = pkd.BatchDecodeWithPagedKVCache(w.hq, w.hkv, w.head_dim, P, max_batch=w.batch,
                                                max_num_pages=_nnz(name, tables),
                                                shared_prefix=gi is not None and not cascade,
                                                cascade=cascade,
                                                kv_dtype=w.kv_dtype,
                                                kv_layout=w.kv_layout,
                                                num_pages=w.pool_pages,
                                                use_tensor_cores={"auto": None, "fma": False,
                                                                  "mma": True}[args.consumer],
                                                chunk_rule=args.chunk_rule, alpha=args.alpha,
                                                dense_prefix=(gi is not None and not cascade
                                                              and args.prefix_kernel == "dense"),
                                                device=dev)
            _plan(d, gi, tables, name=name)
            decs.append(d)
        sets.append(decs)
    decs = sets[0]
    # graphs: per context, one per cache copy; each captures the layers of a
    # step.  `graphs` are the plain graphs of the timed steps; `tgraphs` carry
    # CUDA event nodes around every decode launch for the per-kernel roofline
    # (event nodes break the kernel-to-kernel programmatic launch overlap, so
    # they are kept out of the step timing).
    graphs = [[] for _ in range(n_sets)]
    tgraphs = [[] for _ in range(n_sets)]
    if cascade:
        # one context: the cascade launch and its merge, per cache copy
        for si, ds in enumerate(sets):
            for c in range(copies):
                for timing, dst in ((False, graphs), (True, tgraphs)):
                    dst[si].append((ds[0].capture([qs[0]], [kvs[c]], [outs[0]], [lses[0]],
                                                  timing=timing), None, c))
    elif w.prefix_tokens:
        # prefix run + suffix run + merge_states, per cache copy.  The step
        # graph holds all three: the two levels are independent and run on
        # two captured streams, merge_states joins them.  The timing graphs
        # (event nodes around each decode launch) keep the levels apart.
        po = [torch.empty_like(qs[0]) for _ in range(copies)]
        pl = [torch.empty(w.batch, w.hq, dtype=torch.float32, device=dev) for _ in range(copies)]
        so = [torch.empty_like(qs[0]) for _ in range(copies)]
        sl = [torch.empty(w.batch, w.hq, dtype=torch.float32, device=dev) for _ in range(copies)]
        side = torch.cuda.Stream(device=dev)
        for si, ds in enumerate(sets):
            for c in range(copies):
                gp = ds[0].capture([qs[0]], [kvs[c]], [po[c]], [pl[c]], timing=True)
                gs = ds[1].capture([qs[0]], [kvs[c]], [so[c]], [sl[c]], timing=True)
                tgraphs[si].append((gp, gs, c))
                graphs[si].append((_composed_step_graph(ds, qs[0], kvs[c], po[c], pl[c], so[c],
                                                        sl[c], outs[0], lses[0], side, dev),
                                   None, c))
    else:
        for si, ds in enumerate(sets):
            for c in range(copies):
                kv_c = kvs[c * layers:(c + 1) * layers]
                for timing, dst in ((False, graphs), (True, tgraphs)):
                    dst[si].append((ds[0].capture(qs, kv_c, outs, lses, timing=timing,
                                                  kv_scales=kv_scales), None, c))

    stream = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(n_sets)]
    done = [torch.cuda.Event() for _ in range(n_sets)]
    for e in done:
        e.record(stream)

    use = {"graphs": graphs, "eager": args.launch == "eager"}
    if w.prefix_tokens and not cascade:
        fork = torch.cuda.Event()

    def launch_eager(si, c):
        """The step's kernels launched on the stream directly (no graph).
        Each run passes its plan's epoch: the kernels wait on the device for
        that schedule, so no event orders the copy stream's upload before
        them and the step's first kernel may start under the previous
        step's last (programmatic dependent launch)."""
        ds = sets[si]
        if w.prefix_tokens and not cascade:
            fork.record(stream)
            side.wait_event(fork)
            ds[0].run(qs[0], kvs[c], out=po[c], lse=pl[c], stream=stream, expect_epoch=ds[0].epoch)
            ds[1].run(qs[0], kvs[c], out=so[c], lse=sl[c], stream=side, expect_epoch=ds[1].epoch)
            stream.wait_stream(side)
            pkd.merge_states(po[c], pl[c], so[c], sl[c], outs[0], lses[0])
            return
        for l in range(layers):
            ks, vs = kv_scales[l] if kv_scales else (1.0, 1.0)
            ds[0].run(qs[l], kvs[c * layers + l], out=outs[l], lse=lses[l], k_scale=ks,
                      v_scale=vs, stream=stream, expect_epoch=ds[0].epoch)

    def graph_of(k):
        return use["graphs"][k % n_sets][(k // n_sets) % copies]

    def step(k):
        """One decode step on device-resident q / out / lse."""
        si = k % n_sets
        copy_stream.wait_event(done[si])
        for (name, gi, table), d in zip(views, sets[si]):
            _plan(d, gi, table, stream=copy_stream, name=name)
        copied[si].record(copy_stream)
        gp, gs, c = graph_of(k)
        if use["eager"]:
            launch_eager(si, c)
        else:
            stream.wait_event(copied[si])
            gp.launch()
            if gs is not None:   # timing graphs of the shared-prefix step
                gs.launch()
                pkd.merge_states(po[c], pl[c], so[c], sl[c], outs[0], lses[0])
        done[si].record(stream)

    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize()
    # --launch auto: a short untimed trial of both launch modes on this
    # machine (after the warm-up, before the timed steps); the faster one is
    # timed.  Single-layer steps of a few tens of microseconds are close to
    # host-bound with per-step launches, so which mode wins depends on the
    # host; the trial times are reported with the choice.
    launch_trial = None
    chosen = args.launch
    if args.launch == "auto":
        n_trial = max(10, min(args.steps // 2, 100))
        launch_trial = {}
        idx = args.warmup
        for mode in ("graph", "eager"):
            use["eager"] = mode == "eager"
            for _ in range(3):
                step(idx)
                idx += 1
            torch.cuda.synchronize()
            t0e = torch.cuda.Event(enable_timing=True)
            t1e = torch.cuda.Event(enable_timing=True)
            t0e.record(stream)
            for _ in range(n_trial):
                step(idx)
                idx += 1
            t1e.record(stream)
            torch.cuda.synchronize()
            launch_trial[mode] = round(max_over_ranks(t0e.elapsed_time(t1e) / n_trial, world,
                                                      dev), 5)
        chosen = "eager" if launch_trial["eager"] <= launch_trial["graph"] else "graph"
        use["eager"] = chosen == "eager"
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    gpu_uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    sampler = ClockSampler(f"GPU-{gpu_uuid}" if gpu_uuid else dev.index)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with sampler:
        time.sleep(0.3)
        torch.cuda.synchronize()
        e0.record(stream)
        for k in range(args.steps):
            step(args.warmup + k)
        e1.record(stream)
        torch.cuda.synchronize()
    ms_total = e0.elapsed_time(e1)
    # second timed loop, same steps with the event-node graphs: decode-kernel
    # duration of every launch of the last step
    use["graphs"] = tgraphs
    use["eager"] = False
    k_roof = max(3, min(args.steps, 10))
    for k in range(k_roof):
        step(args.warmup + args.steps + k)
    torch.cuda.synchronize()
    last = graph_of(args.warmup + args.steps + k_roof - 1)
    k1_ms = last[0].layer_times() + (last[1].layer_times() if last[1] is not None else [])
    use["graphs"] = graphs
    use["eager"] = chosen == "eager"
    ms_total = max_over_ranks(ms_total, world, dev)
    ms_step = ms_total / args.steps

    # algorithmic bytes of one step
    if w.prefix_tokens:
        n_pre = w.prefix_tokens // w.page_size
        suf_lens = list(w.suffix_lens)
        kv_bytes = (w.prefix_tokens + sum(suf_lens)) * 2 * w.hkv * w.head_dim * 2  # prefix once
        io = w.batch * w.hq * (w.head_dim * 2 * 2 + 4)
        table = 4 * (n_pre + 3 + 2 + int(t["suffix"][0][-1]) + 2 * w.batch + 1)
        step_bytes = kv_bytes + io + table
        if cascade:   # one launch moves the whole step
            layer_bytes = [step_bytes]
        else:
            # per launch: the prefix level reads the shared pages once for all requests
            layer_bytes = [alg_bytes_per_layer(w, [w.prefix_tokens], n_pre),
                           alg_bytes_per_layer(w, suf_lens, int(t["suffix"][0][-1]))]
    else:
        lb = alg_bytes_per_layer(w, lens, nnz)
        step_bytes = lb * layers
        layer_bytes = [lb] * layers
    gbs = aggregate_throughput(step_bytes, ms_step, world)
    peak, peak_kind = measured_peak()
    # roofline of the dominant kernel (decode), per launch
    k1_gbs = [b / (ms * 1e-3) / 1e9 for b, ms in zip(layer_bytes, k1_ms) if ms > 0]
    k1_mean_ms = float(np.mean(k1_ms))
    achieved = float(np.sum(layer_bytes) / (np.sum(k1_ms) * 1e-3) / 1e9)
    info = decs[0].plan_info()

    # end to end: host q in, host out back, plan from host tables, per step
    if cascade:
        side_e2e = [torch.cuda.Stream(device=dev) for _ in range(2)]

        def capture_io(si, dq, do, dl, hq, ho, hl, c):
            nx = 1 - si
            return _cascade_step_graph(
                sets[si][0], dq[si][0], kvs[c], do[si][0], dl[si][0], dev,
                io=((side_e2e[0], side_e2e[1]), [(dq[nx][0], hq[0])],
                    [(ho[0], do[nx][0]), (hl[0], dl[nx][0])]))
        e2e = run_e2e_graph_io(args, sets, views, capture_io, copies, qs, outs, lses, stream,
                               step_bytes, world, dev,
                               kernels="the cascade launch (both levels) + its merge")
    elif w.prefix_tokens:
        side_e2e = [torch.cuda.Stream(device=dev) for _ in range(3)]

        def capture_io(si, dq, do, dl, hq, ho, hl, c):
            # step of set si: computes on set si's q / out / lse while the
            # next step's q goes into the other set's buffer and the previous
            # step's results come back from it
            nx = 1 - si
            return _composed_step_graph(
                sets[si], dq[si][0], kvs[c], po[c], pl[c], so[c], sl[c], do[si][0], dl[si][0],
                side_e2e[0], dev,
                io=((side_e2e[1], side_e2e[2]), [(dq[nx][0], hq[0])],
                    [(ho[0], do[nx][0]), (hl[0], dl[nx][0])]))
        e2e = run_e2e_graph_io(args, sets, views, capture_io, copies, qs, outs, lses, stream,
                               step_bytes, world, dev)
    else:
        def capture(si, dq, do, dl, c):
            return sets[si][0].capture(dq, kvs[c * layers:(c + 1) * layers], do, dl,
                                       kv_scales=kv_scales)
        e2e = run_e2e_pipelined(args, sets, views, capture, copies, qs, outs, lses, stream,
                                step_bytes, world, dev)

    clocks = sampler.summary()
    gp0, _, _ = graphs[0][0]
    launches_per_step = 5 if (w.prefix_tokens and not cascade) else 2 * gp0.layers
    line = {
        "metric": METRIC,
        "value": round(gbs, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "steps_per_s": round(1e3 / ms_step, 3),
        "pct_of_peak": round(100.0 * gbs / world / peak, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.kv_dtype == "bf16" else "e4m3 KV (f16 MMA)",
        "accum_dtype": "fp32",
        "data": "synthetic (seeded N(0,1) bf16 q/KV, seeded lengths and page permutation)",
        "config": {
            "workload": args.workload, "kv_dtype": w.kv_dtype, "kv_layout": w.kv_layout,
            "layers": layers,
            "batch": w.batch, "hq": w.hq,
            "hkv": w.hkv, "head_dim": w.head_dim, "page_size": P,
            "total_tokens_per_layer": int(sum(lens)), "pages_per_layer": nnz,
            "alg_bytes_per_step": int(step_bytes),
            "consumer": args.consumer,
            "chunk_rule": args.chunk_rule,
            "alpha": args.alpha if args.alpha >= 0 else "default (32)",
            "prefix_kernel": (("cascade (dense tensor-core prefix role + decode role, one "
                               "launch, one merge)") if cascade else args.prefix_kernel)
                             if w.prefix_tokens else None,
            "l2": (f"inputs larger than L2: {n_kv} distinct caches of "
                   f"{kvs[0].numel() * kvs[0].element_size() / 1e9:.2f} GB, "
                   + ("one per layer" if copies == 1 else "rotated over replays")),
            "plan": {k: info[k] for k in ("num_ctas", "chunk_tokens", "num_items", "num_units",
                                          "makespan", "prefix_ctas", "prefix_chunk_tokens")},
            "launch": ("step graphs replayed (one per cache copy and planning context), "
                       "each after an event on the step's schedule upload"
                       if chosen == "graph" else
                       "kernels launched on the stream per step; they wait on the device for "
                       "their plan's schedule (pkd_run with expect_epoch), no event")
                      + (f"; chosen by --launch auto from an untimed trial of "
                         f"{launch_trial} ms per step" if launch_trial else ""),
            "parallelism": f"replicas x{world} (no collective)",
        },
        "roofline": {
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
            "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
            else "fallback",
            "unit": "GB/s", "frac": round(achieved / peak, 4),
            "traffic": traffic_from_profile(args.workload,
                                            "cascade_kernel" if cascade else "decode_kernel"),
            "kernel": "cascade_kernel" if cascade else "decode_kernel",
            "launch_ms_mean": round(k1_mean_ms, 5),
            "launch_gbs_min": round(min(k1_gbs), 1) if k1_gbs else None,
            "launch_gbs_max": round(max(k1_gbs), 1) if k1_gbs else None,
            "timing": "CUDA event nodes around each decode launch inside a replayed copy of "
                      "the step graph, in a second timed loop of the same steps (last step); "
                      "the step time comes from the first loop",
        },
        "e2e": e2e,
        "gpu_launches": int(launches_per_step * args.steps),
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, t, qs, kvs, budget_s=args.cpu_seconds)
    return line


def run_e2e_pipelined(args, sets, views, capture, copies, qs, outs, lses, stream, step_bytes,
                      world, dev):
    """The step through the public API with host buffers, the way a serving
    loop pipelines it: step k's queries go host -> device on a copy stream
    (DMA engines) while step k-1's graph runs, and step k's out + lse go back
    on a second copy stream while step k+1 runs.  The two planning contexts
    each own a set of device q / out / lse buffers, so no copy touches a
    buffer a running graph uses.  Every step still moves its own inputs in
    and its own results out inside the timed region (the last step's results
    are on the host when it ends).  capture(set, q, out, lse, cache copy)
    returns the step graph of a planning context over those buffers."""
    import torch
    n_sets = len(sets)
    hq = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in qs]
    for h, x in zip(hq, qs):
        h.copy_(x)
    ho = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in outs]
    hl = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in lses]
    dq = [[torch.empty_like(x) for x in qs] for _ in range(n_sets)]
    do = [[torch.empty_like(x) for x in outs] for _ in range(n_sets)]
    dl = [[torch.empty_like(x) for x in lses] for _ in range(n_sets)]
    graphs = [[capture(si, dq[si], do[si], dl[si], c) for c in range(copies)]
              for si in range(n_sets)]
    h2d_stream = torch.cuda.Stream(device=dev)
    d2h_stream = torch.cuda.Stream(device=dev)
    ready = [torch.cuda.Event() for _ in range(n_sets)]   # inputs + plan of the set's step
    ran = [torch.cuda.Event() for _ in range(n_sets)]     # the set's graph finished
    back = [torch.cuda.Event() for _ in range(n_sets)]    # its results are on the host
    for si in range(n_sets):
        ran[si].record(stream)
        back[si].record(stream)

    def step(k):
        si = k % n_sets
        # the set's buffers are free once its previous graph ran and its
        # results went back
        h2d_stream.wait_event(ran[si])
        h2d_stream.wait_event(back[si])
        for (name, gi, table), d in zip(views, sets[si]):
            _plan(d, gi, table, stream=h2d_stream, name=name)
        with torch.cuda.stream(h2d_stream):
            for x, h in zip(dq[si], hq):
                x.copy_(h, non_blocking=True)
            ready[si].record(h2d_stream)
        stream.wait_event(ready[si])
        graphs[si][(k // n_sets) % copies].launch()
        ran[si].record(stream)
        d2h_stream.wait_event(ran[si])
        with torch.cuda.stream(d2h_stream):
            for x, h in zip(do[si], ho):
                h.copy_(x, non_blocking=True)
            for x, h in zip(dl[si], hl):
                h.copy_(x, non_blocking=True)
            back[si].record(d2h_stream)

    h2d = sum(x.numel() * x.element_size() for x in qs)
    d2h = sum(x.numel() * x.element_size() for x in outs) + sum(x.numel() * 4 for x in lses)
    sched = sum(4 * d.plan_info()["schedule_words"] for d in sets[0])
    steps = max(3, args.steps // 2)
    for k in range(3):
        step(k)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(stream)
    for k in range(steps):
        step(k)
    stream.wait_stream(d2h_stream)
    e1.record(stream)
    torch.cuda.synchronize()
    wall = (time.perf_counter() - t0) * 1e3 / steps
    gpu_ms = e0.elapsed_time(e1) / steps
    ms = max(gpu_ms, wall)
    for row in graphs:
        for g in row:
            g.close()
    ms = max_over_ranks(ms, world, dev)
    return {"value": round(world * step_bytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(ms, 5), "ms_gpu_events": round(gpu_ms, 5),
            "ms_host_wall": round(wall, 5), "h2d_bytes_per_step": int(h2d + sched),
            "d2h_bytes_per_step": int(d2h),
            "what": "pinned host q -> device (copy stream), plan from host tables (schedule "
                    "H2D), graph replay, out + lse -> pinned host (copy stream); steps "
                    "pipelined over two buffer sets; KV cache resident"}


def run_e2e_graph_io(args, sets, views, capture_io, copies, qs, outs, lses, stream, step_bytes,
                     world, dev, kernels="both levels + merge_states"):
    """The step through the public API with host buffers, for steps short
    enough that per-call host work would bound a loop that issues every copy
    itself: one graph per step runs the step's kernels on one set of device
    q / out / lse buffers and, on two branches beside them, copies the next
    step's q from pinned host memory into the other set and the previous
    step's out + lse from the other set back to pinned host memory.  The
    first step's q goes in before the loop's first graph and the last step's
    results come back after its last one, both inside the timed region, so
    every timed step moves its own inputs in and its own results out.  A step
    costs the host its plan calls (into alternating planning contexts: a
    context's schedule is rewritten only after the step that read it is
    done) and one graph launch.  capture_io(set, device q / out / lse sets,
    host q / out / lse, cache copy) returns such a graph."""
    import torch
    n_sets = len(sets)
    assert n_sets == 2
    hq = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in qs]
    for h, x in zip(hq, qs):
        h.copy_(x)
    ho = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in outs]
    hl = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in lses]
    dq = [[torch.empty_like(x) for x in qs] for _ in range(n_sets)]
    do = [[torch.empty_like(x) for x in outs] for _ in range(n_sets)]
    dl = [[torch.empty_like(x) for x in lses] for _ in range(n_sets)]
    graphs = [[capture_io(si, dq, do, dl, hq, ho, hl, c) for c in range(copies)]
              for si in range(n_sets)]
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(n_sets)]
    done = [torch.cuda.Event() for _ in range(n_sets)]
    for e in done:
        e.record(stream)

    def step(k):
        si = k % n_sets
        copy_stream.wait_event(done[si])
        for (name, gi, table), d in zip(views, sets[si]):
            _plan(d, gi, table, stream=copy_stream, name=name)
        copied[si].record(copy_stream)
        stream.wait_event(copied[si])
        graphs[si][(k // n_sets) % copies].launch()
        done[si].record(stream)

    def prologue():
        with torch.cuda.stream(stream):
            for x, h in zip(dq[0], hq):
                x.copy_(h, non_blocking=True)

    def epilogue(last):
        with torch.cuda.stream(stream):
            for x, h in zip(do[last % n_sets], ho):
                h.copy_(x, non_blocking=True)
            for x, h in zip(dl[last % n_sets], hl):
                h.copy_(x, non_blocking=True)

    h2d = sum(x.numel() * x.element_size() for x in qs)
    d2h = sum(x.numel() * x.element_size() for x in outs) + sum(x.numel() * 4 for x in lses)
    sched = sum(4 * d.plan_info()["schedule_words"] for d in sets[0])
    steps = max(4, args.steps // 2) // 2 * 2
    prologue()
    for k in range(4):
        step(k)
    epilogue(3)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(stream)
    prologue()
    for k in range(steps):
        step(k)
    epilogue(steps - 1)
    e1.record(stream)
    torch.cuda.synchronize()
    wall = (time.perf_counter() - t0) * 1e3 / steps
    gpu_ms = e0.elapsed_time(e1) / steps
    ms = max(gpu_ms, wall)
    for row in graphs:
        for g in row:
            g.close()
    ms = max_over_ranks(ms, world, dev)
    return {"value": round(world * step_bytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(ms, 5), "ms_gpu_events": round(gpu_ms, 5),
            "ms_host_wall": round(wall, 5), "h2d_bytes_per_step": int(h2d + sched),
            "d2h_bytes_per_step": int(d2h),
            "what": "plan from host tables (schedule H2D on a copy stream), then one graph "
                    f"per step: {kernels} on one buffer set while the next "
                    "step's q (pinned host -> device) and the previous step's out + lse "
                    "(device -> pinned host) move on two branches beside them; the first q "
                    "and the last results are copied inside the timed region too; KV cache "
                    "resident"}


# ------------------------------------------------------------ cpu baseline

def _oracle_sample(w, t, q_bits, kv_bits, rows_req, nthreads=None):
    import oracle
    rows = np.array([(i, h) for i in rows_req for h in range(w.hq)], dtype=np.int32)
    t0 = time.perf_counter()
    if w.kv_dtype == "e4m3":
        s = workloads.FP8_AMAX / 448.0
        oracle.attend_fp8(q_bits, kv_bits, t["indptr"], t["indices"], t["last"], rows,
                          hq=w.hq, hkv=w.hkv, k_scale=s, v_scale=s, nthreads=nthreads,
                          layout=w.kv_layout)
    else:
        oracle.attend(q_bits, kv_bits, t["indptr"], t["indices"], t["last"], rows,
                      hq=w.hq, hkv=w.hkv, nthreads=nthreads, layout=w.kv_layout)
    return time.perf_counter() - t0


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the
    machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def cpu_baseline(w, t, qs, kvs, budget_s=12.0, q_bits=None, kv_bits=None):
    """The fp64 oracle on the host cores, on a bounded sample of the same
    workload (requests of layer 0, all query heads), in the metric's unit."""
    import oracle
    from oracle import _bits, _u8
    oracle.build()
    if q_bits is None:
        q_bits = _bits(qs[0])
        kv_bits = _u8(kvs[0]) if w.kv_dtype == "e4m3" else _bits(kvs[0])
    lens = _lens(t, w.page_size)
    order = list(range(w.batch))
    # calibrate on one request; the sample is requests 0, 1, ... of layer 0,
    # cycling through the layer as many times as the time budget allows
    def sample_for(budget, nthreads):
        t_one = _oracle_sample(w, t, q_bits, kv_bits, [order[0]], nthreads)
        n_tok_target = budget / max(t_one / max(lens[order[0]], 1), 1e-9)
        sample, acc = [], 0
        while acc < n_tok_target and len(sample) < 64 * w.batch:
            i = order[len(sample) % w.batch]
            sample.append(i)
            acc += lens[i]
        return sample

    def gbs(sample, secs):
        s_lens = [lens[i] for i in sample]
        bytes_ = alg_bytes_per_layer(
            workloads.Workload("s", 0, w.hq, w.hkv, w.head_dim, w.page_size, 1, tuple(s_lens), 1,
                               kv_dtype=w.kv_dtype),
            s_lens, sum(-(-l // w.page_size) for l in s_lens))
        return bytes_ / secs / 1e9

    # the same sample timed three times (a third of the budget each): median
    sample = sample_for(budget_s / 3.0, None)
    runs = sorted(_oracle_sample(w, t, q_bits, kv_bits, sample) for _ in range(3))
    secs = runs[1]
    passes = len(sample) / w.batch
    # one host core, on a sample a sixth of the budget long
    sample1 = sample_for(budget_s / 6.0, 1)
    secs1 = _oracle_sample(w, t, q_bits, kv_bits, sample1, 1)
    return {"value": round(gbs(sample, secs), 4), "unit": "GB/s", "cores": os.cpu_count(),
            "cpu_model": cpu_model(),
            "kind": "oracle", "seconds": round(secs, 3),
            "runs_s": [round(x, 3) for x in runs], "statistic": "median of 3",
            "sample": f"layer 0: {len(sample)} request rows ({passes:.2f} passes over the "
                      f"{w.batch} requests, {sum(lens[i] for i in sample)} tokens) x {w.hq} "
                      f"query heads, fp64, all host cores",
            "single_core": {"value": round(gbs(sample1, secs1), 4), "unit": "GB/s", "cores": 1,
                            "seconds": round(secs1, 3),
                            "sample": f"layer 0: {len(sample1)} request rows x {w.hq} query "
                                      f"heads, fp64, one thread"}}


# The Composable Format latency table of the pages (FlashInfer 完全拆解,
# Composable Format 只在复用足够大时占优): (shared prefix tokens, batch) with
# 128-token suffixes, and their microseconds for the composable and the single
# format (FP16, GPU of that paper, not stated per table) -- context only.
PREFIX_GRID = [(1024, 16, 45.17, 46.52), (8192, 16, 88.67, 226.57), (32768, 16, 217.42, 945.67),
               (1024, 64, 87.86, 130.49), (8192, 64, 125.76, 931.75), (32768, 64, 254.54, 4090.0)]


# Short shared prefixes around the point where the cascade stops paying
# (not in the pages' table): the format advice is checked on them too.
EXTRA_PREFIX_CASES = [(16, 16, None, None), (128, 16, None, None), (256, 16, None, None),
                      (16, 64, None, None), (128, 64, None, None)]


def run_prefix_sweep(args, rank, world):
    """Shared prefix, composable against single format, over the pages' grid.
    Composable: the prefix level planned once for the whole batch (the dense
    tcgen05 kernel reads the prefix once per KV head) and the suffix level,
    on two streams, joined by merge_states -- one CUDA graph.  Cascade: both
    levels in one plan, one launch (dense prefix CTAs beside decode CTAs)
    and one merge.  Single: every request over its full page table (prefix
    pages then its own), one decode + merge.  GPU time per step, back to
    back, rotating over enough cache copies that the step's bytes are not
    L2-resident; the host plans once per case (its cost is not in these
    numbers).  Eager launches by default: replaying one captured graph per
    cache copy adds a cost per launch that grows with the number of distinct
    graphs replayed in turn (about 20 us per step at 160), whatever memory
    they read."""
    import torch

    import paged_kv_decode_host_gb300 as pkd

    pkd.build()
    pkd.load()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream(device=dev)
    reps = max(args.steps, 20) if args.launch == "graph" else min(max(args.steps, 20), 200)
    rows = []
    launches = 0
    grid = PREFIX_GRID + EXTRA_PREFIX_CASES
    if args.sweep_cases:
        want = {tuple(int(x) for x in c.split("x")) for c in args.sweep_cases.split(",")}
        grid = [row for row in grid if (row[0], row[1]) in want]
        if not grid:
            raise SystemExit(f"--sweep-cases {args.sweep_cases}: no such (prefix x batch)")
    for prefix, B, pages_comp, pages_single in grid:
        w = workloads.shared_prefix_case(prefix, B)
        t = workloads.make_tables(w)
        P = w.page_size
        n_pre = prefix // P
        pool_bytes = w.pool_pages * 2 * P * w.hkv * w.head_dim * 2
        copies = max(2, int(np.ceil(1.2e9 / pool_bytes)))
        kvs = workloads.make_kv(w, device=dev, layers=copies)
        q = workloads.make_q(w, device=dev, layers=1)[0]
        mk = lambda **kw: pkd.BatchDecodeWithPagedKVCache(w.hq, w.hkv, w.head_dim, P,
                                                         max_batch=B, num_pages=w.pool_pages,
                                                         device=dev, **kw)
        pre = mk(max_num_pages=n_pre, shared_prefix=True, dense_prefix=True)
        pre.plan_shared(np.array([0, B], np.int32), np.array([0, n_pre], np.int32),
                        np.asarray(t["prefix"][1][:n_pre], np.int32), np.array([P], np.int32))
        suf = mk(max_num_pages=int(t["suffix"][0][-1]))
        suf.plan(*t["suffix"])
        single = mk(max_num_pages=int(t["indptr"][-1]))
        single.plan(t["indptr"], t["indices"], t["last"])
        gi = np.array([0, B], np.int32)
        prefix_t = (np.array([0, n_pre], np.int32), np.asarray(t["prefix"][1][:n_pre], np.int32),
                    np.array([P], np.int32))
        casc = mk(max_num_pages=n_pre + int(t["suffix"][0][-1]), cascade=True)
        casc.plan_cascade(gi, prefix_t, t["suffix"])
        po, so, out_c, out_s, out_k = (torch.empty_like(q) for _ in range(5))
        pl, sl, lse_c, lse_s, lse_k = (torch.empty(B, w.hq, dtype=torch.float32, device=dev)
                                       for _ in range(5))
        if args.launch == "graph":
            comp = [_composed_step_graph((pre, suf), q, kvs[c], po, pl, so, sl, out_c, lse_c,
                                         side, dev).launch for c in range(copies)]
            sing = [single.capture([q], [kvs[c]], [out_s], [lse_s]).launch
                    for c in range(copies)]
            cgr = [casc.capture([q], [kvs[c]], [out_k], [lse_k]).launch for c in range(copies)]
        else:
            fork = torch.cuda.Event()

            def composed(c):
                def f():
                    fork.record(stream)
                    side.wait_event(fork)
                    pre.run(q, kvs[c], out=po, lse=pl, stream=stream)
                    suf.run(q, kvs[c], out=so, lse=sl, stream=side)
                    stream.wait_stream(side)
                    pkd.merge_states(po, pl, so, sl, out_c, lse_c)
                return f
            comp = [composed(c) for c in range(copies)]
            sing = [lambda c=c: single.run(q, kvs[c], out=out_s, lse=lse_s, stream=stream)
                    for c in range(copies)]
            cgr = [lambda c=c: casc.run(q, kvs[c], out=out_k, lse=lse_k, stream=stream)
                   for c in range(copies)]
        us = {}
        for name, gs in (("composable", comp), ("single", sing), ("cascade", cgr)):
            for k in range(3):
                gs[k % copies]()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            if args.launch != "graph":
                # the host queues the steps while the stream sleeps, so the
                # events time the GPU's work back to back, not the host's
                torch.cuda._sleep(int(4e7))
            e0.record(stream)
            for k in range(reps):
                gs[k % copies]()
            e1.record(stream)
            torch.cuda.synchronize()
            us[name] = e0.elapsed_time(e1) * 1e3 / reps
        # the two formats compute the same states (up to rounding)
        comp[0]()
        sing[0]()
        cgr[0]()
        torch.cuda.synchronize()
        diff = float(max((out_c.float() - out_s.float()).abs().max(),
                         (out_k.float() - out_s.float()).abs().max()))
        ldiff = float(max((lse_c - lse_s).abs().max(), (lse_k - lse_s).abs().max()))
        launches += reps * (5 + 2 + 2)
        cinfo = casc.plan_info()
        acfg = pkd.make_config(w.hq, w.hkv, w.head_dim, P, B, n_pre + int(t["suffix"][0][-1]),
                               w.pool_pages, -1, -1, cinfo["num_ctas"], pkd.FLAG_CASCADE)
        advice = pkd.advise_format(acfg, gi, prefix_t, t["suffix"])
        auto = "cascade" if advice["use_cascade"] else "single"
        kv_once = (prefix + 128 * B) * 2 * w.hkv * w.head_dim * 2
        rows.append({"prefix": prefix, "batch": B, "suffix": 128,
                     "composable_us": round(us["composable"], 2),
                     "cascade_us": round(us["cascade"], 2),
                     "single_us": round(us["single"], 2),
                     "speedup": round(us["single"] / us["composable"], 2),
                     "cascade_speedup": round(us["single"] / us["cascade"], 2),
                     "cascade_plan": {k: cinfo[k] for k in ("prefix_ctas", "prefix_chunk_tokens",
                                                            "chunk_tokens", "num_items")},
                     "advice": {"format": auto, "cascade_us": round(advice["cascade_us"], 1),
                                "single_us": round(advice["single_us"], 1),
                                "cascade_makespan": advice["cascade_makespan"],
                                "single_makespan": advice["single_makespan"]},
                     "auto_us": round(us[auto], 2),
                     "auto_vs_best": round(us[auto] / min(us.values()), 3),
                     "composable_GBps_prefix_once": round(kv_once / (us["composable"] * 1e3), 1),
                     "single_GBps_per_request_reads": round(
                         (prefix + 128) * B * 2 * w.hkv * w.head_dim * 2 / (us["single"] * 1e3), 1),
                     "max_abs_diff_out": round(diff, 5), "max_abs_diff_lse": round(ldiff, 6),
                     "pages_us_composable": pages_comp, "pages_us_single": pages_single,
                     "cache_copies": copies})
        del kvs, comp, sing, cgr, pre, suf, single, casc
        torch.cuda.empty_cache()
    big = [r for r in rows if r["prefix"] == 32768 and r["batch"] == 64] or rows[-1:]
    big = big[0]
    return {"metric": "shared-prefix decode latency, composable vs single format "
                      "(GPU us per step)",
            "value": big["composable_us"], "unit": "us", "n_gpus": world, "steps": reps,
            "warmup": 3, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16 q/KV, scattered pages)",
            "config": {"workload": "prefix_sweep", "hq": 32, "hkv": 8, "head_dim": 128,
                       "page_size": 16, "suffix": 128,
                       "l2": "cache copies rotated per step, >= 1.2 GB in total",
                       "launch": ("CUDA-graph replays, one graph per cache copy"
                                  if args.launch == "graph" else
                                  "kernels launched on the stream, queued behind a GPU sleep "
                                  "so that the events time the GPU's work back to back")},
            "table": rows, "gpu_launches": launches,
            "note": "pages_us_*: the pages' table (FP16, other GPU), context only"}


def run_append(args, rank, world):
    """append_paged_kv_cache for the Llama-shaped step: each of the 64
    requests appends its new token (K and V rows, all 8 KV heads) into its
    page slot, in each of the 32 layer caches.  One step = one CUDA-graph
    replay of one every-layer append launch (pkd_append_kv_layers); the
    per-layer form (32 launches per step, one graph) is timed beside it.
    Bytes: the new rows read + written and the table words read."""
    import torch

    import paged_kv_decode_host_gb300 as pkd

    pkd.build()
    pkd.load()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = workloads.workload("llama8b_step")
    t = workloads.make_tables(w)
    lens = _lens(t, w.page_size)
    B, L = w.batch, w.layers
    kvs = workloads.make_kv(w, device=dev, layers=L)
    g = torch.Generator(device=dev).manual_seed(77)
    k_new = [torch.randn(B, w.hkv, w.head_dim, generator=g, device=dev).to(torch.bfloat16)
             for _ in range(L)]
    v_new = [torch.randn(B, w.hkv, w.head_dim, generator=g, device=dev).to(torch.bfloat16)
             for _ in range(L)]
    as_dev = lambda a: torch.tensor(np.asarray(a, dtype=np.int32), device=dev)
    bidx, pos = as_dev(range(B)), as_dev([l - 1 for l in lens])
    ip, ix, la = as_dev(t["indptr"]), as_dev(t["indices"]), as_dev(t["last"])
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def step_layers():
        pkd.append_kv_layers(k_new, v_new, bidx, pos, ip, ix, la, kvs, err=err)

    def step_per_layer():
        for l in range(L):
            pkd.append_kv(k_new[l], v_new[l], bidx, pos, ip, ix, la, kvs[l], err=err)

    def graph_of(fn):
        fn()
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            fn()
        for _ in range(args.warmup):
            gr.replay()
        torch.cuda.synchronize()
        return gr

    def time_graph(gr):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            gr.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    graph, graph_pl = graph_of(step_layers), graph_of(step_per_layer)
    gpu_uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    sampler = ClockSampler(f"GPU-{gpu_uuid}" if gpu_uuid else dev.index)
    with sampler:
        time.sleep(0.3)
        ms = time_graph(graph)
    ms_pl = time_graph(graph_pl)
    assert int(err.item()) == 0
    row = w.hkv * w.head_dim * 2
    step_bytes = L * (B * 2 * row * 2 + 4 * (2 * B + 2 * B + 1 + B))
    peak, peak_kind = measured_peak()
    gbs = world * step_bytes / (ms * 1e-3) / 1e9
    return {
        "metric": "append_paged_kv_cache throughput (new K/V rows into page slots)",
        "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "per_layer_launches": {"ms_per_step": round(ms_pl, 5),
                               "us_per_launch": round(1e3 * ms_pl / L, 3),
                               "GBps": round(world * step_bytes / (ms_pl * 1e-3) / 1e9, 2)},
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "append", "layers": L, "batch": B, "hkv": w.hkv,
                   "head_dim": w.head_dim, "page_size": w.page_size,
                   "bytes_per_step": int(step_bytes), "launch": "one every-layer launch"},
        "roofline": {"bound": "latency (16.8 MB per launch)", "achieved": round(gbs, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4),
                     "traffic": None},
        "gpu_launches": args.steps, "clocks": sampler.summary(),
    }


def run_reference_append(args, world):
    """Reference arm for the append workload: the numpy append oracle on one
    layer of the Llama-shaped step (64 new tokens)."""
    import torch
    from oracle import _bits
    from oracle import append as oappend
    w = workloads.workload("llama8b_step")
    t = workloads.make_tables(w)
    lens = _lens(t, w.page_size)
    kv = _bits(workloads.make_kv(w, device="cpu", layers=1)[0])
    g = torch.Generator().manual_seed(77)
    k_new = _bits(torch.randn(w.batch, w.hkv, w.head_dim, generator=g).to(torch.bfloat16))
    row = w.hkv * w.head_dim * 2
    layer_bytes = w.batch * 2 * row * 2 + 4 * (5 * w.batch + 1)
    secs = []
    for k in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oappend.append_kv(kv, k_new, k_new, range(w.batch), [l - 1 for l in lens], t["indptr"],
                          t["indices"], t["last"], w.page_size)
        if k >= args.warmup:
            secs.append(time.perf_counter() - t0)
    v = layer_bytes / float(np.mean(secs)) / 1e9
    return {"impl": "reference", "metric": "append_paged_kv_cache throughput (new K/V rows into "
            "page slots)", "value": round(v, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * float(np.mean(secs)), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 bits", "data": "synthetic",
            "config": {"workload": "append", "sample_per_step": "one layer (64 tokens)"},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": "one layer (64 tokens), numpy, one core"},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def run_reference(args, rank, world):
    """Reference arm: the fp64 CPU oracle, as it stands, on the host cores."""
    import torch
    if args.workload == "append":
        return run_reference_append(args, world)
    if args.workload == "prefix_sweep":
        raise SystemExit("the reference arm times the oracle on one workload at a time; "
                         "prefix_sweep is a table of GPU timings")
    w = workloads.workload(args.workload)
    t = workloads.make_tables(w)
    from oracle import _bits, _u8
    q = workloads.make_q(w, device="cpu", layers=1)[0]
    # only the pages the sample touches need values; build the whole layer
    if w.kv_dtype == "e4m3":
        kv = workloads.make_kv_fp8(w, device="cpu", layers=1)[0][0]
        kv_bits = _u8(kv)
    else:
        kv = workloads.make_kv(w, device="cpu", layers=1)[0]
        kv_bits = _bits(kv)
    q_bits = _bits(q)
    del kv
    per_step_budget = max(1.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    lens = _lens(t, w.page_size)
    for _ in range(args.warmup):
        cpu_baseline(w, t, None, None, budget_s=per_step_budget, q_bits=q_bits, kv_bits=kv_bits)
    vals, secs = [], 0.0
    last = None
    for _ in range(args.steps):
        last = cpu_baseline(w, t, None, None, budget_s=per_step_budget, q_bits=q_bits,
                            kv_bits=kv_bits)
        vals.append(last["value"])
        secs += last["seconds"]
    v = float(np.mean(vals))
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * secs / max(args.steps, 1), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": args.workload, "layers": w.layers, "batch": w.batch, "hq": w.hq,
                   "hkv": w.hkv, "head_dim": w.head_dim, "page_size": w.page_size,
                   "sample_per_step": last["sample"] if last else None},
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": os.cpu_count(),
                         "cpu_model": cpu_model(), "kind": "oracle",
                         "sample": last["sample"] if last else None},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# ------------------------------------------------------- other workloads

# The other synthetic configurations a decode step is quoted on, timed in the
# same process after the headline: the 63 + 100,000-token skewed batch, the
# page-size-1 token-sparse batch and the shared-prefix step.
OTHER_WORKLOADS = ("skewed", "token_sparse", "shared_prefix")


def _child_env(local_rank):
    """Environment for a single-process bench run on this rank's GPU."""
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "LOCAL_WORLD_SIZE", "MASTER_ADDR",
                        "MASTER_PORT", "GROUP_RANK", "ROLE_RANK", "TORCHELASTIC_RUN_ID")}
    visible = os.environ.get("CUDA_VISIBLE_DEVICES")
    devs = [d for d in visible.split(",") if d.strip()] if visible else None
    env["CUDA_VISIBLE_DEVICES"] = devs[local_rank] if devs else str(local_rank)
    return env


def run_other_workloads(args, rank, world, names=OTHER_WORKLOADS):
    """Each workload as its own bench run (same timing, roofline and e2e
    legs, no CPU baseline), summarised under one key of the headline line.
    Each runs in a fresh process on this rank's GPU, as it would standalone:
    in a process that has already run other workloads the per-step host
    work (planning, launches) ran measurably slower, and the single-layer
    steps are short enough for the host to matter.  With several ranks,
    every rank runs its own and the whole-job figures take the slowest."""
    import gc

    import torch
    gc.collect()
    torch.cuda.empty_cache()
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    dev = torch.device("cuda", local_rank)
    res = {}
    for name in names:
        cmd = [sys.executable, os.path.abspath(__file__), "--workload", name,
               "--steps", str(args.other_steps), "--warmup", str(max(args.warmup, 10)),
               "--no-other-workloads", "--no-cpu-baseline", "--launch", args.launch,
               "--consumer", args.consumer, "--chunk-rule", args.chunk_rule,
               "--alpha", str(args.alpha), "--prefix-mode", args.prefix_mode,
               "--prefix-kernel", args.prefix_kernel]
        r = subprocess.run(cmd, env=_child_env(local_rank), capture_output=True, text=True,
                           cwd=ROOT)
        lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
        if r.returncode != 0 or not lines:
            raise RuntimeError(f"{name} bench run failed ({r.returncode}): {r.stderr[-2000:]}")
        ln = json.loads(lines[-1])
        step_bytes = ln["config"]["alg_bytes_per_step"]
        ms = max_over_ranks(ln["ms_per_step"], world, dev)
        e2e = dict(ln["e2e"])
        e2e_ms = max_over_ranks(e2e["ms_per_step"], world, dev)
        if world > 1:
            e2e["value"] = round(aggregate_throughput(step_bytes, e2e_ms, world), 2)
            e2e["ms_per_step"] = round(e2e_ms, 5)
        rf = ln["roofline"]
        value = aggregate_throughput(step_bytes, ms, world)
        res[name] = {
            "value": round(value, 2), "unit": ln["unit"],
            "pct_of_peak": round(100.0 * value / world / rf["peak"], 2),
            "ms_per_step": round(ms, 5), "steps_per_s": round(1e3 / ms, 3),
            "steps": ln["steps"], "warmup": ln["warmup"],
            "roofline": {k: rf[k] for k in ("bound", "achieved", "peak", "frac", "traffic",
                                            "launch_ms_mean")},
            "e2e": {k: e2e[k] for k in ("value", "unit", "ms_per_step", "ms_gpu_events",
                                        "ms_host_wall", "h2d_bytes_per_step",
                                        "d2h_bytes_per_step")},
            "clocks": ln["clocks"], "gpu_launches": ln["gpu_launches"],
            "config": {k: ln["config"][k] for k in ("batch", "hq", "hkv", "page_size",
                                                    "total_tokens_per_layer",
                                                    "alg_bytes_per_step", "l2", "plan",
                                                    "prefix_kernel", "launch")},
            "process": "own (a bench.py run of this workload alone on this GPU)",
        }
    return res


# --------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama8b_step",
                    choices=["llama8b_step", "skewed", "token_sparse", "shared_prefix",
                             "llama8b_step_fp8", "llama8b_step_hnd", "llama8b_step_fp8_hnd",
                             "shared_prefix_hnd", "append", "prefix_sweep"])
    ap.add_argument("--consumer", choices=["auto", "fma", "mma"], default="auto",
                    help="decode-kernel consumer: the default, or forced CUDA-core (fma) / "
                         "tensor-core (mma) folding of the GQA group")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--chunk-rule", choices=["closed", "search"], default="closed",
                    help="split chunk: closed-form work bound (default) or the largest chunk "
                         "that still gives every CTA an item (binary search)")
    ap.add_argument("--sweep-cases", default="",
                    help="prefix_sweep: only these cases, e.g. 32768x64,1024x16 (prefix x batch)")
    ap.add_argument("--alpha", type=int, default=-1,
                    help="planner per-item cost in tokens (cost = alpha + tokens); -1: default")
    ap.add_argument("--launch", choices=["auto", "graph", "eager"], default="auto",
                    help="timed steps: launch the step's kernels on the stream, each run "
                         "waiting on the device for its plan's schedule (pkd_run with "
                         "expect_epoch; the upload goes on a copy stream with no event), or "
                         "replay the step's captured CUDA graphs (one per cache copy and "
                         "planning context) after an event on the upload; auto: whichever "
                         "an untimed trial after the warm-up finds faster on this machine "
                         "(prefix_sweep: auto is eager)")
    ap.add_argument("--prefix-mode", choices=["cascade", "levels"], default="cascade",
                    help="shared-prefix step: one cascade plan and launch with one merge, or "
                         "two levels (prefix context + suffix context) joined by merge_states")
    ap.add_argument("--prefix-kernel", choices=["dense", "mma"], default="dense",
                    help="shared-prefix level: the tcgen05 dense kernel (128-row tiles per KV "
                         "head) or the mma.sync row-block consumer (16-row tiles)")
    ap.add_argument("--layers", type=int, default=0,
                    help="layers per step (0: the workload's own); smaller for profiling captures")
    ap.add_argument("--copies", type=int, default=0,
                    help="cache copies rotated by single-layer workloads (0: enough for 1.2 GB); "
                         "fewer only to keep profiling captures small")
    ap.add_argument("--other-steps", type=int, default=300,
                    help="timed steps of each other workload reported with the default one")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="report the selected workload alone")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    if args.workload == "append":
        line = run_append(args, rank, world)
    elif args.workload == "prefix_sweep":
        line = run_prefix_sweep(args, rank, world)
    else:
        line = run_ours(args, rank, world)
        if (args.workload == "llama8b_step" and args.layers == 0 and
                not args.no_other_workloads):
            line["other_workloads"] = run_other_workloads(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
