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
import re
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
    ap.add_argument("--config", type=int, default=1,
                    help="workload index 0..4 (1 = pure decode); 5 = speculative verification")
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
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the configured workload (no per_config block)")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def make_workload(config: int, rank: int = 0, reqs=None, seed_offset: int = 0):
    """Replica `rank` of workload `config`: same shapes, its own seed."""
    import workloads as W
    base = {0: 1000, 1: 1001, 2: 1002, 3: 1003, 4: 1004, 5: 1006}[config] + 7919 * (rank + seed_offset)
    if config == 0:
        return W.toy_r1r2(base)
    if config == 1:
        return W.pure_decode(base, **({} if reqs is None else {"num_reqs": reqs}))
    if config == 2:
        return W.mixed_step(base, **({} if reqs is None else {"n_decode": reqs}))
    if config == 3:
        return W.long_context(base, **({} if reqs is None else {"num_reqs": reqs}))
    if config == 5:  # beyond the five: speculative verification, 4 rows per request
        return W.spec_decode(base, **({} if reqs is None else {"num_reqs": reqs}))
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


def request_kv_lens(step) -> np.ndarray:
    """Keys of the last cross row of each request with a row (its seq_len)."""
    qsl = np.asarray(step.query_start_loc, dtype=np.int64)
    q_len = np.diff(qsl)
    want = np.ones_like(q_len) if step.rows_per_req is None else np.asarray(step.rows_per_req)
    k = np.minimum(np.maximum(want, 0), np.maximum(q_len, 0))
    seq = np.asarray(step.seq_lens, dtype=np.int64)
    return np.maximum(seq[k > 0], 0)


def accounting(wl, step, e4m3: bool = False) -> dict:
    """Algorithmic bytes of one step (per layer and per step). With an e4m3 cache
    the keys/values take one byte each and every page read adds its 16-byte
    scale record; queries and outputs stay in the workload's dtype."""
    from workloads import elem_bytes
    sz = elem_bytes(wl.dtype)
    kv_sz = 1 if e4m3 else sz
    kv = cross_rows_kv_lens(step)
    rows = int(kv.shape[0])
    # logical bytes (the metric): every row reads its own causal prefix
    kv_bytes_layer = int(kv.sum()) * 2 * wl.num_kv_heads * wl.head_dim * kv_sz
    # algorithmic bytes (the roofline): the rows of a request share its pages, read
    # once up to the last row's end (seq_len keys); one row per request: the same
    last = request_kv_lens(step)
    uniq_kv_bytes_layer = int(last.sum()) * 2 * wl.num_kv_heads * wl.head_dim * kv_sz
    qo_bytes_layer = 2 * rows * wl.num_q_heads * wl.head_dim * sz
    page_meta = 4 + (16 if e4m3 else 0)
    bt_bytes_layer = page_meta * int(np.sum((last + wl.block_size - 1) // wl.block_size)) * \
        wl.num_kv_heads
    # read + write
    append_bytes = 2 * step.num_tokens * wl.num_kv_heads * wl.head_dim * (sz + kv_sz)
    return {
        "rows": rows,
        "kv_bytes_layer": kv_bytes_layer,
        "attn_bytes_layer": uniq_kv_bytes_layer + qo_bytes_layer + bt_bytes_layer,
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


def _code_only(text: str) -> str:
    """C++/CUDA source without its comments and blank lines."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = []
    for line in text.splitlines():
        cut = line.find("//")
        if cut >= 0:
            line = line[:cut]
        if line.strip():
            out.append(line.rstrip())
    return "\n".join(out)


def kernel_source_sha() -> str:
    """Hash of the code the dominant kernel is built from (comments and blank
    lines left out: editing a comment does not change the kernel)."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "yoco_shared_kv_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
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


def _graph_time_ms(g, stream, reps, warm=3):
    """Average replay time of CUDA graph g on `stream` (CUDA events, after warm-up)."""
    import torch
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(warm):
            g.replay()
        c0.record(stream)
        for _ in range(reps):
            g.replay()
        c1.record(stream)
    stream.synchronize()
    return c0.elapsed_time(c1) / reps


def cold_layer_ms(dw, ds, cq, stream, dev, reps):
    """One layer (layer 0) from an L2 that holds none of the cache, two ways.

    clean: the L2 is first filled by READING a buffer of 2 x L2 (a reduction),
    so it holds only clean, unrelated lines; the layer's DRAM traffic is its own.
    dirty: the L2 is first filled by WRITING 2 x L2 (a memset); the layer then
    also pays for writing back the ~L2 of dirty lines it evicts.
    Each is graph(flush, layer 0) minus graph(flush), CUDA events."""
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.zeros(2 * l2 // 4, dtype=torch.int32, device=dev)
    sink = torch.zeros((), dtype=torch.int64, device=dev)
    out = {}
    for kind in ("clean", "dirty"):
        def fl():
            if kind == "clean":
                torch.sum(flush, dim=0, out=sink)
            else:
                flush.zero_()
        g_fl, g_cold = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_fl, stream=stream):
            fl()
        with torch.cuda.graph(g_cold, stream=stream):
            fl()
            dw.attend(ds, 0, cq=cq)
        t_fl = _graph_time_ms(g_fl, stream, reps)
        t_cold = _graph_time_ms(g_cold, stream, reps)
        out[kind] = max(t_cold - t_fl, 1e-6)
        del g_fl, g_cold
    del flush
    return out


def measure(args, config, rank, world, local, *, kv="native", fused=False, steps=None,
            warmup=None, e2e=True, cold=True, l2_window=False, alternate=True, reqs=None,
            seed_offset=0):
    """Time one workload through the whole path on this rank's GPU.

    Returns the record of one bench line (without clocks or the CPU baseline):
    the step's logical KV GB/s, query rows/s, the dominant kernel's launch
    figures, one layer from a cold L2, and the end-to-end figure with host
    copies."""
    import torch
    from yoco_shared_kv_gb300 import _native as N
    from yoco_shared_kv_gb300 import pipeline as P

    steps = args.steps if steps is None else steps
    warmup = args.warmup if warmup is None else warmup
    dev = torch.device("cuda", local)
    wl = make_workload(config, rank, reqs, seed_offset)
    e4m3 = kv == "e4m3"
    if e4m3 and wl.dtype != "bf16":
        return None
    if e4m3:
        from workloads import page_scales
        dw = P.DeviceWorkload(wl, dev, pin_host=e2e, sentinel=False, kv="e4m3",
                              page_scales=page_scales(wl))
    else:
        dw = P.DeviceWorkload(wl, dev, pin_host=e2e, sentinel=False)
    if not alternate:
        dw.alternate = False
    step_i = len(wl.steps) - 1
    ds = dw.steps[step_i]
    acc = accounting(wl, wl.steps[step_i], e4m3)
    workload_name = wl.name + ("_e4m3kv" if e4m3 else "")
    if fused and not dw.decode_only(step_i):
        raise SystemExit("--fused needs a decode-only workload (one token and one row per request)")

    def step_fn_on(d_s):
        if fused:
            dw.fused_step_on(d_s)
        else:
            dw.run_step_on(d_s)
    stream = torch.cuda.Stream(device=dev)
    if l2_window:  # before capture: the kernel nodes take the stream's window
        N.yoco_set_l2_window(dw.k_cache, dw.k_cache.numel() * dw.k_cache.element_size(), -1.0,
                             stream=stream)
    with torch.cuda.stream(stream):
        dw.run_fill(stream)
        for i in range(step_i):  # earlier steps of a multi-step schedule
            dw.run_step(i, stream)
    stream.synchronize()

    # our kernels per step: append and selection (unless fused), the step's
    # plan (tensor-core paths), and per layer one attention kernel (the fp32
    # path adds its split merge when the plan has more than one split)
    tc = e4m3 or wl.dtype == "bf16"
    merges = 0 if tc else (1 if N.yoco_cross_attn_workspace_size(
        max(ds.rows_upper, 1), wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size,
        ds.max_seq_len, P.torch_dtype(wl.dtype)) > 0 else 0)
    launches_per_step = (0 if fused else 2) + (1 if tc else 0) + wl.layers * (1 + merges)

    L = wl.layers
    # The step runs as one CUDA graph (append -> select -> every layer), as an
    # engine replays its captured cross-decoder; a second graph holds only the
    # L attention calls, to time the dominant kernel on its own.
    with torch.cuda.stream(stream):
        step_fn_on(ds)  # eager once: one-time host set-up before capture
    stream.synchronize()
    g_step, g_attn = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=stream):
        step_fn_on(ds)
    # the fused step runs no row selection: its cross query_start_loc is query_start_loc
    cq = ds.dev["qsl"] if fused else None
    with torch.cuda.graph(g_attn, stream=stream):
        for layer in range(L):
            dw.attend(ds, layer, cq=cq)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g_step.replay()
    stream.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(steps):
            g_step.replay()
        ev1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize(dev)
    elapsed_ms = ev0.elapsed_time(ev1)
    # dominant kernel: the attention calls alone, same inputs, CUDA events
    reps = max(3, steps // 2)
    attn_launch_ms = _graph_time_ms(g_attn, stream, reps, warm=1) / L
    cold_ms = cold_layer_ms(dw, ds, cq, stream, dev, reps) if cold else None

    max_ms, total_kv_bytes, total_rows = aggregate_ranks(
        elapsed_ms, acc["kv_bytes_step"] * steps, acc["rows"] * L * steps, world, dev)
    if dw.error_bits() != 0:
        raise RuntimeError(f"device error bits {dw.error_bits():#x}")

    # End to end through the C ABI: every step copies its inputs from pinned host
    # memory and reads its outputs back, as a serving loop does. Two buffer sets
    # alternate, so the copies of one step overlap the computation of another
    # (copy-in stream, compute stream, read-back stream, ordered by events); the
    # timed region covers every copy.
    e2e_rec = None
    if e2e:
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
        k_e2e = max(1, min(steps, 200))
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
        e2e_rec = {"value": round(total_kv_bytes / steps / (e2e_ms / 1e3) / 1e9, 3),
                   "unit": "GB/s", "ms_per_step": round(e2e_ms, 4),
                   "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                   "how": "two input/output buffer sets; copies overlap the other set's step"}
        del g_b, ds_b
    if l2_window:
        N.yoco_set_l2_window(None, 0, stream=stream)

    ms_per_step = max_ms / steps
    value = total_kv_bytes / (max_ms / 1e3) / 1e9
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"]
    achieved = acc["attn_bytes_layer"] / (attn_launch_ms / 1e3) / 1e9
    traffic = profiled_traffic(workload_name)

    def cold_rec(ms, how):
        gbs = acc["attn_bytes_layer"] / (ms / 1e3) / 1e9
        return {"launch_ms": round(ms, 5), "achieved_gbs": round(gbs, 2),
                "frac": round(gbs / peak, 4), "how": how}
    res = {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 cache, bf16 q/out, f16 mma" if e4m3 else wl.dtype,
        "data": "synthetic (seeded N(0,1) K/V and queries, random page permutation)",
        "config": workload_config(wl, wl.steps[step_i], acc, world, fused, workload_name),
        "hbm_frac": round(value / peak, 4),
        "query_rows_per_s": round(total_rows / (max_ms / 1e3), 1),
        "roofline": {"kernel": DOMINANT_KERNEL + " (cross-CTA merge inside)", "bound": "hbm",
                     "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     # DRAM-side fraction: the bytes DRAM actually moved per launch
                     # inside the layer sequence (ncu), over the same launch time
                     "dram_frac": (None if traffic is None else
                                   round(traffic / (attn_launch_ms / 1e3) / 1e9 / peak, 4)),
                     "algorithmic_bytes_per_launch": acc["attn_bytes_layer"],
                     "launch_ms": round(attn_launch_ms, 5), "peak_source": peaks["source"]},
        "gpu_launches": launches_per_step * steps,
        "per_layer_cold_l2": None if cold_ms is None else cold_rec(
            cold_ms["clean"], "graph(read 2 x L2 with a reduction, layer 0) minus graph(the "
            "reduction), CUDA events: the L2 holds only clean lines of another buffer"),
        "per_layer_cold_l2_dirty": None if cold_ms is None else cold_rec(
            cold_ms["dirty"], "graph(memset 2 x L2, layer 0) minus graph(memset): the layer "
            "also writes back the dirty lines it evicts"),
    }
    if e2e_rec is not None:
        res["e2e"] = e2e_rec
    res["_wl"] = wl
    res["_step_i"] = step_i
    del g_step, g_attn, dw, ds
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return res


def _compact(r: dict) -> dict:
    """The per-workload figures of a measure() record, for the per_config block."""
    if r is None:
        return None
    out = {"workload": r["config"]["workload"], "value": r["value"], "unit": r["unit"],
           "ms_per_step": r["ms_per_step"], "hbm_frac": r["hbm_frac"],
           "query_rows_per_s": r["query_rows_per_s"], "steps": r["steps"],
           "roofline": {k: r["roofline"][k] for k in ("achieved", "frac", "dram_frac",
                                                      "traffic", "launch_ms")}}
    for k in ("per_layer_cold_l2", "per_layer_cold_l2_dirty"):
        if r.get(k):
            out[k] = {"frac": r[k]["frac"], "achieved_gbs": r[k]["achieved_gbs"],
                      "launch_ms": r[k]["launch_ms"]}
    if r.get("e2e"):
        out["e2e"] = {"value": r["e2e"]["value"], "ms_per_step": r["e2e"]["ms_per_step"]}
    if r.get("cpu_baseline"):
        out["cpu_baseline"] = r["cpu_baseline"]
    return out


def run_ours(args, rank, world, local):
    import torch
    from yoco_shared_kv_gb300 import build as B
    if rank == 0 or not os.path.exists(B.LIB):
        B.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.set_device(local)

    sampler = None if args.no_clocks else ClockSampler(local)
    if sampler:
        sampler.mark_start()
    res = measure(args, args.config, rank, world, local, kv=args.kv, fused=args.fused,
                  e2e=not args.no_e2e, cold=not args.no_cold, l2_window=args.l2_window,
                  alternate=not args.no_alternate, reqs=args.reqs, seed_offset=args.seed_offset)
    if sampler:
        sampler.mark_stop()
    wl, step_i = res.pop("_wl"), res.pop("_step_i")
    e4m3 = args.kv == "e4m3"
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not e4m3:
        res["cpu_baseline"] = cpu_baseline(wl, step_i)
    del wl

    # Every workload of the problem statement, the 8-bit cache and the fused
    # decode step, each timed the same way (fewer steps), so that one default
    # run observes them all; the headline above is the configured workload.
    if not args.no_per_config and args.reqs is None and world == 1:
        sub_steps = max(3, min(args.steps, 30))
        sub_warm = max(3, min(args.warmup, 5))
        per = {}
        for c in range(5):
            if c == args.config and not args.fused and args.kv == "native":
                r = dict(res)
            else:
                r = measure(args, c, rank, world, local, steps=sub_steps, warmup=sub_warm,
                            e2e=not args.no_e2e, cold=not args.no_cold)
                wl_c, si = r.pop("_wl"), r.pop("_step_i")
                if rank == 0 and not args.no_cpu_baseline:
                    r["cpu_baseline"] = cpu_baseline(wl_c, si, budget_s=3.0, one_thread_s=1.5)
                del wl_c
            per[str(c)] = _compact(r)
        res["per_config"] = per
        e8 = {}
        for c in range(1, 5):
            r = measure(args, c, rank, world, local, kv="e4m3", steps=sub_steps,
                        warmup=sub_warm, e2e=False, cold=not args.no_cold)
            r.pop("_wl"), r.pop("_step_i")
            e8[str(c)] = _compact(r)
        res["per_config_e4m3"] = e8
        fu = {}
        for kv in ("native", "e4m3"):
            r = measure(args, 1, rank, world, local, kv=kv, fused=True, steps=sub_steps,
                        warmup=sub_warm, e2e=False, cold=False)
            r.pop("_wl"), r.pop("_step_i")
            fu[kv] = {"workload": r["config"]["workload"], "ms_per_step": r["ms_per_step"],
                      "value": r["value"], "query_rows_per_s": r["query_rows_per_s"]}
        res["fused_decode_step"] = fu
        # beyond the five: speculative verification (4 cross rows per request) at
        # the pure-decode shapes
        r = measure(args, 5, rank, world, local, steps=sub_steps, warmup=sub_warm, e2e=False,
                    cold=not args.no_cold)
        r.pop("_wl"), r.pop("_step_i")
        res["multi_row"] = _compact(r)
    res["clocks"] = sampler.stop() if sampler else None
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


def cpu_baseline(wl, step_i: int, budget_s: float = 20.0, one_thread_s: float = 5.0) -> dict:
    """The oracle timed on this host's cores over a bounded sample of the step.

    Sample: every cross row, layers taken one at a time (each with the step's
    append and selection) until `budget_s` is spent, on all host cores; then
    rows of layer 0 one at a time on one thread until `one_thread_s` is spent."""
    import oracle
    step = wl.steps[step_i]
    acc = accounting(wl, step)
    nthreads = host_cores()
    Ks, Vs = _oracle_setup(wl, step)
    kp, vp = wl.empty_pool(), wl.empty_pool()
    kv_lens = cross_rows_kv_lens(step)
    t0 = time.perf_counter()
    done = 0
    for layer in range(wl.layers):
        oracle_step(wl, step, Ks, Vs, kp, vp, nthreads, layers=[layer])
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    kv_bytes = acc["kv_bytes_layer"] * done
    per_key = 2 * wl.num_kv_heads * wl.head_dim * (4 if wl.dtype == "f32" else 2)
    _, cqsl, _ = oracle.select_cross_rows(step.query_start_loc, step.rows_per_req)
    q0 = oracle.widen(step.q[0], wl.dtype)
    t1 = time.perf_counter()
    rows1 = 0
    bytes1 = 0
    for n in range(int(kv_lens.shape[0])):
        oracle.cross_attn(q0, Ks, Vs, step.seq_lens, cqsl, wl.scale, rows=[n], nthreads=1)
        rows1 += 1
        bytes1 += int(kv_lens[n]) * per_key
        if time.perf_counter() - t1 > one_thread_s:
            break
    dt1 = time.perf_counter() - t1
    return {"value": round(kv_bytes / dt / 1e9, 4), "unit": "GB/s", "cores": nthreads,
            "kind": "oracle",
            "sample": f"{acc['rows']} rows x {done} of {wl.layers} layers of {wl.name} "
                      f"(sum kv_len {int(kv_lens.sum())}), float64, {dt:.1f} s",
            "query_rows_per_s": round(acc["rows"] * done / dt, 3),
            "one_thread": {"value": round(bytes1 / dt1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                           "query_rows_per_s": round(rows1 / dt1, 3),
                           "sample": f"{rows1} rows of layer 0, attention only, {dt1:.1f} s"}}


def workload_config(wl, step, acc, world, fused=False, workload_name=None) -> dict:
    """The `config` dict of a bench line (both arms print it for the same workload)."""
    return {
        "workload": workload_name or wl.name, "description": wl.description,
        "H_q": wl.num_q_heads, "H_kv": wl.num_kv_heads, "head_dim": wl.head_dim,
        "block_size": wl.block_size, "layers": wl.layers, "requests": step.num_reqs,
        "step_tokens": step.num_tokens, "cross_rows": acc["rows"],
        "kv_bytes_per_layer": acc["kv_bytes_layer"],
        "l2": ("inputs larger than L2" if acc["kv_bytes_layer"] > 129e6
               else "inputs fit in L2 (layers re-read them: logical bytes)"),
        "parallelism": f"replicas x{world}",
        "step": ("append fused into layer 0 (yoco_cross_decode_step)" if fused
                 else "append, select, every layer"),
    }


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
        "config": workload_config(wl, step, acc, world),
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
