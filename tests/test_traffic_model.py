"""The traffic model (host C function) against the benchmark's accounting and
against DRAM bytes ncu measured for the attention kernel."""
import os

import numpy as np
import pytest
import torch

from tests.conftest import ROOT


@pytest.fixture(scope="module")
def N():
    from yoco_shared_kv_gb300 import build
    build.build()
    from yoco_shared_kv_gb300 import _native
    return _native


def _model(N, wl, st):
    from yoco_shared_kv_gb300.pipeline import torch_dtype
    return N.yoco_cross_decoder_bytes(st.query_start_loc, st.rows_per_req, st.seq_lens, wl.layers,
                                      wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size,
                                      torch_dtype(wl.dtype))


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_model_equals_bench_accounting(N, idx):
    import bench
    from workloads import SMALL
    wl = SMALL[idx]()
    for st in wl.steps:
        tot, per = _model(N, wl, st)
        assert tot == bench.accounting(wl, st)["attn_bytes_layer"] * wl.layers
        assert per.sum() == tot


def test_model_counts_rows_like_selection(N):
    from workloads import chunked_prefill_spec
    wl = chunked_prefill_spec()
    st = wl.steps[0]  # A: non-final chunk -> no row, so no bytes
    tot, per = _model(N, wl, st)
    assert per[0] == 0 and per[1] > 0 and per[2] > 0
    # three speculative rows see 201, 202, 203 keys: they share the request's pages,
    # read once up to 203 keys, and each has its own query and output
    D, H_kv, H_q, bs, L = wl.head_dim, wl.num_kv_heads, wl.num_q_heads, wl.block_size, wl.layers
    exp = (203 * 2 * H_kv * D * 2 + 3 * 2 * H_q * D * 2 + 4 * -(-203 // bs) * H_kv) * L
    assert per[2] == exp
    # the same request with one row: only the queries and outputs of two rows fewer
    rpr = np.asarray(st.rows_per_req).copy()
    rpr[2] = 1
    one, _ = N.yoco_cross_decoder_bytes(st.query_start_loc, rpr, st.seq_lens,
                                        wl.layers, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                        wl.block_size, torch.bfloat16)
    assert tot - one == 2 * 2 * H_q * D * 2 * L


def test_model_predicts_measured_dram_bytes(N):
    """profiles/traffic.txt holds ncu DRAM bytes per attention launch at full size; a launch
    measured alone (caches flushed, no reuse between layers) reads what the model predicts
    (its writes add the workspace partials of the cross-CTA merge, ~1% of the bytes),
    including the speculative workload, whose rows share their request's pages."""
    import bench
    lines = open(os.path.join(ROOT, "profiles", "traffic.txt")).read().splitlines()
    meas = dict(l.split("=", 1) for l in lines if "=" in l and not l.startswith("#"))
    # 5: four rows per request, grouped on one walk: the request's pages are read once
    for cfg, name, e4m3 in ((1, "pure_decode_bf16", False), (3, "long_context_bf16", False),
                            (1, "pure_decode_bf16_e4m3kv", True),
                            (3, "long_context_bf16_e4m3kv", True), (5, "spec_decode_bf16", False)):
        wl = bench.make_workload(cfg)
        st = wl.steps[-1]
        dt = torch.float8_e4m3fn if e4m3 else torch.bfloat16
        tot, _ = N.yoco_cross_decoder_bytes(st.query_start_loc, st.rows_per_req, st.seq_lens,
                                            wl.layers, wl.num_q_heads, wl.num_kv_heads,
                                            wl.head_dim, wl.block_size, dt)
        per_layer = tot / wl.layers
        assert per_layer == bench.accounting(wl, st, e4m3)["attn_bytes_layer"]
        assert abs(float(meas[name + "_isolated_read"]) / per_layer - 1.0) < 0.006, name  # within 0.6 %
        assert float(meas[name + "_isolated"]) / per_layer < 1.015, name  # partials: < 1.5 % more
        # inside the layer sequence part of it comes from L2 (layers alternate walk direction)
        assert float(meas[name]) < float(meas[name + "_isolated"])


def test_model_rejects_bad_arguments(N):
    with pytest.raises(ValueError):
        N.yoco_cross_decoder_bytes([0, 3, 2], None, [5, 5], 1, 8, 2, 128, 16, torch.bfloat16)
