"""Shared test plumbing: run a workload on the GPU path and on the oracle."""
from __future__ import annotations

import os

import numpy as np

import oracle

ATOL = {"f32": 2e-3, "bf16": 2e-2}  # max |gpu - oracle| (bf16: bf16 output, fp32 accumulation)


def host_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_pools(wl):
    """Pools after the fill and every step, appended by the oracle."""
    kp, vp = wl.empty_pool(), wl.empty_pool()
    for st in ([wl.fill] if wl.fill is not None else []) + wl.steps:
        assert oracle.kv_append(st.k_new, st.v_new, kp, vp, st.block_table, st.seq_lens,
                                st.query_start_loc, wl.block_size) == 0
    return kp, vp


def oracle_step_kv(wl, step):
    Ks, Vs = [], []
    for r in step.req_ids:
        K, V = wl.request_kv(r)
        Ks.append(oracle.widen(K, wl.dtype))
        Vs.append(oracle.widen(V, wl.dtype))
    return Ks, Vs


def oracle_step_out(wl, step, layers=None, rows=None):
    """Oracle attention output [layers, rows, H_q, D] (float64) for one step."""
    _, cqsl, st = oracle.select_cross_rows(step.query_start_loc, step.rows_per_req)
    assert st >= 0
    Ks, Vs = oracle_step_kv(wl, step)
    outs = []
    for layer in (range(wl.layers) if layers is None else layers):
        q = oracle.widen(step.q[layer], wl.dtype)
        o, s = oracle.cross_attn(q, Ks, Vs, step.seq_lens, cqsl, wl.scale, rows=rows,
                                 nthreads=host_threads())
        assert s == 0
        outs.append(o)
    return np.stack(outs)


def gpu_out(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def pool_bits(t) -> np.ndarray:
    """Device pool -> numpy array of its raw element bits."""
    import torch
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.view(torch.int32).cpu().numpy().view(np.uint32)


def oracle_bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint16) if a.dtype == np.uint16 else a.view(np.uint32)


# ------------------------------------------------------------------ e4m3 cache

def oracle_e4m3_pools(wl, scales):
    """e4m3 pools (uint8, sentinel 0xFF) after the fill and every step."""
    kp = np.full(wl.pool_shape(), 0xFF, dtype=np.uint8)
    vp = np.full(wl.pool_shape(), 0xFF, dtype=np.uint8)
    for st in ([wl.fill] if wl.fill is not None else []) + wl.steps:
        assert oracle.kv_append_e4m3(st.k_new, st.v_new, kp, vp, scales, st.block_table,
                                     st.seq_lens, st.query_start_loc, wl.block_size) == 0
    return kp, vp


def oracle_e4m3_step_out(wl, step, kp, vp, scales, layers=None, rows=None):
    """Oracle attention [layers, rows, H_q, D] over the dequantised cache, read back
    through each request's block table."""
    _, cqsl, st = oracle.select_cross_rows(step.query_start_loc, step.rows_per_req)
    assert st >= 0
    Ks, Vs = [], []
    for i in range(step.num_reqs):
        n = int(step.seq_lens[i])
        Ks.append(oracle.e4m3_gather(kp, scales, 0, step.block_table[i], n))
        Vs.append(oracle.e4m3_gather(vp, scales, 1, step.block_table[i], n))
    outs = []
    for layer in (range(wl.layers) if layers is None else layers):
        q = oracle.widen(step.q[layer], wl.dtype)
        o, s = oracle.cross_attn(q, Ks, Vs, step.seq_lens, cqsl, wl.scale, rows=rows,
                                 nthreads=host_threads())
        assert s == 0
        outs.append(o)
    return np.stack(outs)
