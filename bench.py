#!/usr/bin/env python3
"""Benchmark of the YOCO cross-decoder hot path on GB300.

One step = one scheduling step of the workload through the whole path:
yoco_kv_append (the step's new shared K^/V^), yoco_select_cross_rows, then
yoco_cross_attn_paged once per cross-decoder layer against the one shared
cache. Inputs are seeded synthetic data resident in HBM before timing.

Prints one JSON line (rank 0). Metric: KV GB/s read by the cross-decoder
attention (logical bytes: every layer re-reads each row's causal K/V), its
fraction of the measured HBM peak, and query rows/s.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1] [--impl ours|reference]

Under torchrun each rank runs an independent replica (requests are
independent; no collective is on the data path) and the slowest rank's time
is reported.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "cross-decoder paged attn: KV GB/s (% of HBM peak), query rows/s at 1 GB300"
FALLBACK_HBM_GBS = 6800.0
DOMINANT_KERNEL = "attn_tc_persistent"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.txt")


# ------------------------------------------------------------------ helpers


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", type=int, default=1, help="workload index 0..4 (1 = pure decode)")
    ap.add_argument("--reqs", type=int, default=None, help="smaller case: override request count")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-cold", action="store_true", help="skip the cold-L2 single-layer timing")
    ap.add_argument("--l2-window", action="store_true",
                    help="keep part of the K pool persisting in L2 across layers (yoco_set_l2_window)")
    ap.add_argument("--no-alternate", action="store_true",
                    help="every layer walks its pages forward (no cross-layer L2 reuse by direction)")
    ap.add_argument("--seed-offset", type=int, default=0)
    ap.add_argument("--kv", choices=["native", "e4m3"], default="native",
                    help="cache format: the workload's dtype, or e4m3 with per-page scales")
    ap.add_argument("--fused", action="store_true",
                    help="decode workloads: fuse the append into layer 0 (yoco_cross_decode_step)")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def make_workload(config: int, rank: int = 0, reqs=None, seed_offset: int = 0):
    """Replica `rank` of workload `config`: same shapes, its own seed."""
    import workloads as W
    base = {0: 1000, 1: 1001, 2: 1002, 3: 1003, 4: 1004}[config] + 7919 * (rank + seed_offset)
    if config == 0:
        return W.toy_r1r2(base)
    if config == 1:
        return W.pure_decode(base, **({} if reqs is None else {"num_reqs": reqs}))
    if config == 2:
        return W.mixed_step(base, **({} if reqs is None else {"n_decode": reqs}))
    if config == 3:
        return W.long_context(base, **({} if reqs is None else {"num_reqs": reqs}))
    return W.shared_prefix(base, **({} if reqs is None else {"num_reqs": reqs}))


def cross_rows_kv_lens(step) -> np.ndarray:
    """Keys attended by each cross row (accounting only: bytes and rows for the metric)."""
    qsl = np.asarray(step.query_start_loc, dtype=np.int64)
    q_len = np.diff(qsl)
    want = np.ones_like(q_len) if step.rows_per_req is None else np.asarray(step.rows_per_req)
    k = np.minimum(np.maximum(want, 0), np.maximum(q_len, 0))
    lens = []
    for r, kr in enumerate(k):
        for i in range(int(kr)):
            lens.append(int(step.seq_lens[r]) - int(kr) + i + 1)
    return np.asarray(lens, dtype=np.int64)


def accounting(wl, step, e4m3: bool = False) -> dict:
    """Algorithmic bytes of one step (per layer and per step). With an e4m3 cache
    the keys/values take one byte each and every page read adds its 16-byte
    scale record; queries and outputs stay in the workload's dtype."""
    from workloads import elem_bytes
    sz = elem_bytes(wl.dtype)
    kv_sz = 1 if e4m3 else sz
    kv = cross_rows_kv_lens(step)
    rows = int(kv.shape[0])
    kv_bytes_layer = int(kv.sum()) * 2 * wl.num_kv_heads * wl.head_dim * kv_sz
    qo_bytes_layer = 2 * rows * wl.num_q_heads * wl.head_dim * sz
    page_meta = 4 + (16 if e4m3 else 0)
    bt_bytes_layer = page_meta * int(np.sum((kv + wl.block_size - 1) // wl.block_size)) * \
        wl.num_kv_heads
    # read + write
    append_bytes = 2 * step.num_tokens * wl.num_kv_heads * wl.head_dim * (sz + kv_sz)
    return {
        "rows": rows,
        "kv_bytes_layer": kv_bytes_layer,
        "attn_bytes_layer": kv_bytes_layer + qo_bytes_layer + bt_bytes_layer,
        "kv_bytes_step": kv_bytes_layer * wl.layers,
        "append_bytes_step": append_bytes,
        "layers": wl.layers,
    }


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except (OSError, ValueError, KeyError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback"}


KERNEL_SOURCES = ("attn_tc.cuh", "attn_tc.cu", "attn_tc_e4m3.cu", "attn_common.cuh", "common.cuh")


def kernel_source_sha() -> str:
    """Hash of the sources the dominant kernel is built from."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "yoco_shared_kv_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on this workload with the current kernel source."""
    try:
        lines = open(PROFILE_TRAFFIC).read().splitlines()
    except OSError:
        return None
    kv = dict(l.split("=", 1) for l in lines if "=" in l and not l.startswith("#"))
    if kv.get("source_sha") != kernel_source_sha():
        return None
    try:
        return float(kv[workload])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while work runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        self.t_start = self.t_stop = None

    def mark_start(self):
        self.t_start = time.time()

    def mark_stop(self):
        self.t_stop = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for row in csv.reader(io.StringIO(out)):
            if len(row) < 9:
                continue
            try:
                sm.append(float(row[1]))
                smax.append(float(row[2]))
            except ValueError:
                continue
            for nm, v in zip(names, row[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "reasons": sorted(reasons), "samples": len(sm)}


def aggregate_ranks(elapsed_ms: float, kv_bytes: float, rows: float, world: int, device):
    """Whole-job numbers: the slowest rank's time, the units of every rank.

    Replicas share nothing on the data path; this is the only collective.
    """
    if world <= 1:
        return float(elapsed_ms), float(kv_bytes), float(rows)
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed_ms, float(kv_bytes), float(rows)], dtype=torch.float64,
                     device=device)
    tmax = t.clone()
    dist.all_reduce(tmax, op=dist.ReduceOp.MAX)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(tmax[0]), float(t[1]), float(t[2])


# --------------------------------------------------------------- our arm


def run_ours(args, rank, world, local):
    import torch
    from yoco_shared_kv_gb300 import build as B
    if rank == 0 or not os.path.exists(B.LIB):
        B.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    from yoco_shared_kv_gb300 import _native as N
    from yoco_shared_kv_gb300 import pipeline as P

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = make_workload(args.config, rank, args.reqs, args.seed_offset)
    e4m3 = args.kv == "e4m3"
    if e4m3:
        from workloads import page_scales
        dw = P.DeviceWorkload(wl, dev, pin_host=not args.no_e2e, sentinel=False, kv="e4m3",
                              page_scales=page_scales(wl))
    else:
        dw = P.DeviceWorkload(wl, dev, pin_host=not args.no_e2e, sentinel=False)
    if args.no_alternate:
        dw.alternate = False
    step_i = len(wl.steps) - 1
    ds = dw.steps[step_i]
    acc = accounting(wl, wl.steps[step_i], e4m3)
    workload_name = wl.name + ("_e4m3kv" if e4m3 else "")
    if args.fused and not dw.decode_only(step_i):
        raise SystemExit("--fused needs a decode-only workload (one token and one row per request)")

    def step_fn(i):
        step_fn_on(dw.steps[i])

    def step_fn_on(d_s):
        if args.fused:
            dw.fused_step_on(d_s)
        else:
            dw.run_step_on(d_s)
    stream = torch.cuda.Stream(device=dev)
    if args.l2_window:  # before capture: the kernel nodes take the stream's window
        N.yoco_set_l2_window(dw.k_cache, dw.k_cache.numel() * dw.k_cache.element_size(), -1.0,
                             stream=stream)
    with torch.cuda.stream(stream):
        dw.run_fill(stream)
        for i in range(step_i):  # earlier steps of a multi-step schedule
            dw.run_step(i, stream)
    stream.synchronize()

    ws_bytes = ds.workspace.numel() if ds.workspace is not None else 0
    merges = 1 if N.yoco_cross_attn_workspace_size(max(ds.rows_upper, 1), wl.num_q_heads,
                                                   wl.num_kv_heads, wl.head_dim, wl.block_size,
                                                   ds.max_seq_len,
                                                   torch.float8_e4m3fn if e4m3
                                                   else P.torch_dtype(wl.dtype)) > 0 else 0
    launches_per_step = (0 if args.fused else 2) + wl.layers * (1 + merges)

    sampler = None if args.no_clocks else ClockSampler(local)
    L = wl.layers
    # The step runs as one CUDA graph (append -> select -> every layer), as an
    # engine replays its captured cross-decoder; a second graph holds only the
    # L attention calls, to time the dominant kernel on its own.
    with torch.cuda.stream(stream):
        step_fn(step_i)  # eager once: one-time host set-up before capture
    stream.synchronize()
    g_step, g_attn = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=stream):
        step_fn(step_i)
    # the fused step runs no row selection: its cross query_start_loc is query_start_loc
    cq = ds.dev["qsl"] if args.fused else None
    with torch.cuda.graph(g_attn, stream=stream):
        for layer in range(L):
            dw.attend(ds, layer, cq=cq)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g_step.replay()
    stream.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.mark_start()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            g_step.replay()
        ev1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.mark_stop()
    elapsed_ms = ev0.elapsed_time(ev1)
    # dominant kernel: the attention calls alone, same inputs, CUDA events
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    reps = max(3, args.steps // 2)
    with torch.cuda.stream(stream):
        g_attn.replay()
        a0.record(stream)
        for _ in range(reps):
            g_attn.replay()
        a1.record(stream)
    stream.synchronize()
    attn_launch_ms = a0.elapsed_time(a1) / (reps * L)
    # one layer from a cold L2: a graph of (flush, layer 0) minus a graph of the flush alone
    cold_ms = None
    if not args.no_cold:
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
        g_fl, g_cold = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_fl, stream=stream):
            flush.zero_()
        with torch.cuda.graph(g_cold, stream=stream):
            flush.zero_()
            dw.attend(ds, 0, cq=cq)
        times = []
        for g in (g_fl, g_cold):
            c0 = torch.cuda.Event(enable_timing=True)
            c1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                for _ in range(3):
                    g.replay()
                c0.record(stream)
                for _ in range(reps):
                    g.replay()
                c1.record(stream)
            stream.synchronize()
            times.append(c0.elapsed_time(c1) / reps)
        cold_ms = max(times[1] - times[0], 1e-6)
        del flush

    max_ms, total_kv_bytes, total_rows = aggregate_ranks(
        elapsed_ms, acc["kv_bytes_step"] * args.steps, acc["rows"] * L * args.steps, world, dev)
    clocks = sampler.stop() if sampler else None
    if dw.error_bits() != 0:
        raise RuntimeError(f"device error bits {dw.error_bits():#x}")

    # End to end through the C ABI: every step copies its inputs from pinned host
    # memory and reads its outputs back, as a serving loop does. Two buffer sets
    # alternate, so the copies of one step overlap the computation of another
    # (copy-in stream, compute stream, read-back stream, ordered by events); the
    # timed region covers every copy.
    e2e = None
    if not args.no_e2e:
        ds_b = dw.step_buffers(step_i)
        g_b = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            step_fn_on(ds_b)  # eager once, then capture
        stream.synchronize()
        with torch.cuda.graph(g_b, stream=stream):
            step_fn_on(ds_b)
        bufs = [(ds, g_step), (ds_b, g_b)]
        out_host = [torch.empty(b.out.shape, dtype=b.out.dtype, pin_memory=True) for b, _ in bufs]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event() for _ in bufs]
        ev_done = [torch.cuda.Event() for _ in bufs]
        ev_read = [torch.cuda.Event() for _ in bufs]
        k_e2e = max(1, min(args.steps, 200))
        warm = 4
        h2d = d2h = 0
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        for k in range(warm + k_e2e):
            if k == warm:
                torch.cuda.synchronize(dev)
                e0.record(stream)
                s_in.wait_event(e0)
                s_out.wait_event(e0)
            j = k % 2
            dsj, gj = bufs[j]
            if k >= 2:
                s_in.wait_event(ev_done[j])   # the step two back has read these inputs
            with torch.cuda.stream(s_in):
                h2d = dsj.h2d(s_in)
                ev_in[j].record(s_in)
            stream.wait_event(ev_in[j])
            if k >= 2:
                stream.wait_event(ev_read[j])  # and its outputs have been read back
            with torch.cuda.stream(stream):
                gj.replay()
                ev_done[j].record(stream)
            s_out.wait_event(ev_done[j])
            with torch.cuda.stream(s_out):
                out_host[j].copy_(dsj.out, non_blocking=True)
                ev_read[j].record(s_out)
            d2h = out_host[j].numel() * out_host[j].element_size()
        stream.wait_event(ev_read[(warm + k_e2e - 1) % 2])
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = e0.elapsed_time(e1) / k_e2e
        if world > 1:
            import torch.distributed as dist
            t = torch.tensor([e2e_ms], dtype=torch.float64, device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            e2e_ms = float(t[0])
        e2e = {"value": round(total_kv_bytes / args.steps / (e2e_ms / 1e3) / 1e9, 3), "unit": "GB/s",
               "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h),
               "how": "two input/output buffer sets; copies overlap the other set's step"}

    ms_per_step = max_ms / args.steps
    value = total_kv_bytes / (max_ms / 1e3) / 1e9
    peaks = measured_peaks()
    achieved = acc["attn_bytes_layer"] / (attn_launch_ms / 1e3) / 1e9
    traffic = profiled_traffic(workload_name)
    res = {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 cache, bf16 q/out, f16 mma" if e4m3 else wl.dtype,
        "data": "synthetic (seeded N(0,1) K/V and queries, random page permutation)",
        "config": {
            "workload": workload_name, "description": wl.description, "H_q": wl.num_q_heads,
            "H_kv": wl.num_kv_heads, "head_dim": wl.head_dim, "block_size": wl.block_size,
            "layers": wl.layers, "requests": wl.steps[step_i].num_reqs,
            "step_tokens": wl.steps[step_i].num_tokens, "cross_rows": acc["rows"],
            "kv_bytes_per_layer": acc["kv_bytes_layer"],
            "l2": ("inputs larger than L2" if acc["kv_bytes_layer"] > 129e6
                   else "inputs fit in L2 (layers re-read them: logical bytes)"),
            "parallelism": f"replicas x{world}",
            "step": ("append fused into layer 0 (yoco_cross_decode_step)" if args.fused
                     else "append, select, every layer"),
        },
        "hbm_frac": round(value / peaks["hbm_gbs"], 4),
        "query_rows_per_s": round(total_rows / (max_ms / 1e3), 1),
        "roofline": {"kernel": DOMINANT_KERNEL + " (+ split merge)", "bound": "hbm",
                     "achieved": round(achieved, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": acc["attn_bytes_layer"],
                     "launch_ms": round(attn_launch_ms, 5), "peak_source": peaks["source"]},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "per_layer_cold_l2": None if cold_ms is None else {
            "launch_ms": round(cold_ms, 5),
            "achieved_gbs": round(acc["attn_bytes_layer"] / (cold_ms / 1e3) / 1e9, 2),
            "frac": round(acc["attn_bytes_layer"] / (cold_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
            "how": "graph(flush 2 x L2 with a memset, layer 0) minus graph(flush), CUDA events"},
    }
    if e2e is not None:
        res["e2e"] = e2e
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not e4m3:
        res["cpu_baseline"] = cpu_baseline(wl, step_i)
    return res


# ------------------------------------------------------------ oracle (CPU)


def host_cores() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_step(wl, step, Ks, Vs, kp, vp, nthreads, layers=None, rows=None):
    """One step through the CPU oracle: append, select, attention per layer."""
    import oracle
    oracle.kv_append(step.k_new, step.v_new, kp, vp, step.block_table, step.seq_lens,
                     step.query_start_loc, wl.block_size)
    _, cqsl, _ = oracle.select_cross_rows(step.query_start_loc, step.rows_per_req)
    for layer in (range(wl.layers) if layers is None else layers):
        q = oracle.widen(step.q[layer], wl.dtype)
        oracle.cross_attn(q, Ks, Vs, step.seq_lens, cqsl, wl.scale, rows=rows, nthreads=nthreads)


def _oracle_setup(wl, step):
    """Each scheduled request's contiguous K/V, widened for the oracle."""
    import oracle
    Ks, Vs = [], []
    for r in step.req_ids:
        K, V = wl.request_kv(r)
        Ks.append(oracle.widen(K, wl.dtype))
        Vs.append(oracle.widen(V, wl.dtype))
    return Ks, Vs


def cpu_baseline(wl, step_i: int, budget_s: float = 20.0) -> dict:
    """The oracle timed on this host's cores over a bounded sample of the step."""
    step = wl.steps[step_i]
    acc = accounting(wl, step)
    nthreads = host_cores()
    Ks, Vs = _oracle_setup(wl, step)
    kp, vp = wl.empty_pool(), wl.empty_pool()
    kv_lens = cross_rows_kv_lens(step)
    # sample: all rows, layers taken one at a time until the budget is spent
    t0 = time.perf_counter()
    done = 0
    for layer in range(wl.layers):
        oracle_step(wl, step, Ks, Vs, kp, vp, nthreads, layers=[layer])
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    kv_bytes = acc["kv_bytes_layer"] * done
    return {"value": round(kv_bytes / dt / 1e9, 4), "unit": "GB/s", "cores": nthreads,
            "kind": "oracle",
            "sample": f"{acc['rows']} rows x {done} of {wl.layers} layers of {wl.name} "
                      f"(sum kv_len {int(kv_lens.sum())}), float64, {dt:.1f} s",
            "query_rows_per_s": round(acc["rows"] * done / dt, 3)}


def run_reference(args, rank, world):
    """The oracle as the reference arm: same metric/config, host cores, bounded steps."""
    wl = make_workload(args.config, 0, args.reqs, args.seed_offset)
    step_i = len(wl.steps) - 1
    step = wl.steps[step_i]
    acc = accounting(wl, step)
    nthreads = host_cores()
    Ks, Vs = _oracle_setup(wl, step)
    kp, vp = wl.empty_pool(), wl.empty_pool()
    # a reference step is the step's append + select + a bounded number of
    # layers over all rows, sized so the whole run stays within minutes
    t0 = time.perf_counter()
    oracle_step(wl, step, Ks, Vs, kp, vp, nthreads, layers=[0])
    one = time.perf_counter() - t0
    budget_per_step = 120.0 / max(1, args.steps + args.warmup)
    layers = max(1, min(wl.layers, int(budget_per_step / max(one, 1e-6))))
    for _ in range(args.warmup):
        oracle_step(wl, step, Ks, Vs, kp, vp, nthreads, layers=range(layers))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(wl, step, Ks, Vs, kp, vp, nthreads, layers=range(layers))
    dt = time.perf_counter() - t0
    kv_bytes = acc["kv_bytes_layer"] * layers * args.steps
    value = kv_bytes / dt / 1e9
    sample = f"{acc['rows']} rows x {layers} of {wl.layers} layers per step of {wl.name}"
    return {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": wl.name, "description": wl.description},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": nthreads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "query_rows_per_s": round(acc["rows"] * layers * args.steps / dt, 3),
    }


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    res = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
