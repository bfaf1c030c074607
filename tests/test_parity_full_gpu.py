"""The five workloads at full size, in the launch configuration the benchmark
times: append and selection compared bit-exactly (whole pools), attention on
sampled rows and layers against the oracle, plus properties that hold at any
size."""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import ATOL, gpu_out, oracle_bits, oracle_pools, oracle_step_out, pool_bits
from workloads import FULL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def P():
    from yoco_shared_kv_gb300 import build
    build.build()
    from yoco_shared_kv_gb300 import pipeline
    return pipeline


@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_full_size(P, idx):
    wl = FULL[idx]()
    dw = P.DeviceWorkload(wl)
    dw.run_fill()
    dw.run_step(0)
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    step = wl.steps[0]
    ds = dw.steps[0]
    # selection: bit-exact
    o_rows, o_cq, n = oracle.select_cross_rows(step.query_start_loc, step.rows_per_req)
    assert int(ds.num_rows.item()) == n == step.rows_upper
    assert np.array_equal(ds.row_indices.cpu().numpy()[:n], o_rows)
    assert np.array_equal(ds.cqsl.cpu().numpy(), o_cq)
    # append: the whole pool, bit-exact (written slots and untouched sentinel)
    kp, vp = oracle_pools(wl)
    assert np.array_equal(pool_bits(dw.k_cache), oracle_bits(kp))
    assert np.array_equal(pool_bits(dw.v_cache), oracle_bits(vp))
    del kp, vp
    # attention: every output finite; sampled rows x layers against the oracle
    got = gpu_out(ds.out)
    assert np.isfinite(got).all()
    rng = np.random.default_rng(idx)
    rows = sorted(set([0, n - 1] + rng.choice(n, size=min(n, 3), replace=False).tolist()))
    layers = [0, wl.layers - 1]
    ref = oracle_step_out(wl, step, layers=layers, rows=rows)
    sub = got[layers][:, rows]
    err = np.abs(sub - ref).max()
    assert err <= ATOL[wl.dtype], (wl.name, err)
    # layers differ only through their queries: re-running a layer reproduces it exactly
    again = torch.empty_like(ds.out[0])
    dw.attend(ds, 0, out=again)
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int16), ds.out[0].view(torch.int16))


@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_full_size_e4m3(P, idx):
    """The e4m3 cache at full size: quantising append bit-exact over the whole pools,
    attention on sampled rows x layers against the oracle over the dequantised cache."""
    from tests.helpers import oracle_e4m3_pools, oracle_e4m3_step_out
    from workloads import page_scales
    wl = FULL[idx]()
    sc = page_scales(wl)
    dw = P.DeviceWorkload(wl, kv="e4m3", page_scales=sc)
    dw.run_fill()
    dw.run_step(0)
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    step = wl.steps[0]
    ds = dw.steps[0]
    kp, vp = oracle_e4m3_pools(wl, sc)
    assert np.array_equal(dw.k_cache.cpu().numpy(), kp)
    assert np.array_equal(dw.v_cache.cpu().numpy(), vp)
    got = gpu_out(ds.out)
    assert np.isfinite(got).all()
    n = step.rows_upper
    rng = np.random.default_rng(100 + idx)
    rows = sorted(set([0, n - 1] + rng.choice(n, size=min(n, 3), replace=False).tolist()))
    layers = [0, wl.layers - 1]
    ref = oracle_e4m3_step_out(wl, step, kp, vp, sc, layers=layers, rows=rows)
    err = np.abs(got[layers][:, rows] - ref).max()
    assert err <= ATOL["bf16"], (wl.name, err)
    again = torch.empty_like(ds.out[1])
    dw.attend(ds, 1, out=again)  # an odd layer: the reverse page walk at this size
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int16), ds.out[1].view(torch.int16))


@pytest.mark.parametrize("kv", ["native", "e4m3"])
def test_full_size_fused_decode_step(P, kv):
    """Pure decode at full size: the fused step leaves the same cache and the same
    outputs, bit for bit, as the separate append, selection and attention."""
    from workloads import page_scales
    wl = FULL[1]()
    sc = page_scales(wl) if kv == "e4m3" else None
    a = P.DeviceWorkload(wl, kv=kv, page_scales=sc)
    b = P.DeviceWorkload(wl, kv=kv, page_scales=sc)
    for dw in (a, b):
        dw.run_fill()
    a.run_step(0)
    b.fused_step(0)
    torch.cuda.synchronize()
    assert a.error_bits() == 0 and b.error_bits() == 0
    assert torch.equal(a.k_cache.view(torch.uint8), b.k_cache.view(torch.uint8))
    assert torch.equal(a.v_cache.view(torch.uint8), b.v_cache.view(torch.uint8))
    assert torch.equal(a.steps[0].out.view(torch.int16), b.steps[0].out.view(torch.int16))


def test_full_size_speculative_rows(P):
    """Speculative verification at the pure-decode shapes (64 requests x 4 rows):
    selection bit-exact, attention on sampled rows x layers against the oracle."""
    from workloads import MULTI_ROW_FULL
    wl = MULTI_ROW_FULL()
    dw = P.DeviceWorkload(wl)
    dw.run_fill()
    dw.run_step(0)
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    step = wl.steps[0]
    ds = dw.steps[0]
    o_rows, o_cq, n = oracle.select_cross_rows(step.query_start_loc, step.rows_per_req)
    assert n == step.rows_upper == 256
    assert np.array_equal(ds.row_indices.cpu().numpy()[:n], o_rows)
    assert np.array_equal(ds.cqsl.cpu().numpy(), o_cq)
    got = gpu_out(ds.out)
    assert np.isfinite(got).all()
    rng = np.random.default_rng(55)
    rows = sorted(set([0, 1, 2, 3, n - 1] + rng.choice(n, size=4, replace=False).tolist()))
    layers = [0, wl.layers - 1]
    ref = oracle_step_out(wl, step, layers=layers, rows=rows)
    assert np.abs(got[layers][:, rows] - ref).max() <= ATOL["bf16"]


def test_full_size_speculative_rows_e4m3(P):
    """The speculative workload over the e4m3 cache at full size: the 16-wide row
    groups on warp pairs; sampled rows x layers against the oracle over the dequantised
    cache, and an odd layer (backward walk) recomputed bit for bit."""
    from tests.helpers import oracle_e4m3_pools, oracle_e4m3_step_out
    from workloads import MULTI_ROW_FULL, page_scales
    wl = MULTI_ROW_FULL()
    sc = page_scales(wl)
    dw = P.DeviceWorkload(wl, kv="e4m3", page_scales=sc)
    dw.run_fill()
    dw.run_step(0)
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    step = wl.steps[0]
    ds = dw.steps[0]
    kp, vp = oracle_e4m3_pools(wl, sc)
    got = gpu_out(ds.out)
    assert np.isfinite(got).all()
    n = step.rows_upper
    rng = np.random.default_rng(56)
    rows = sorted(set([0, 1, 2, 3, n - 1] + rng.choice(n, size=4, replace=False).tolist()))
    layers = [0, wl.layers - 1]
    ref = oracle_e4m3_step_out(wl, step, kp, vp, sc, layers=layers, rows=rows)
    assert np.abs(got[layers][:, rows] - ref).max() <= ATOL["bf16"]
    again = torch.empty_like(ds.out[1])
    dw.attend(ds, 1, out=again)
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int16), ds.out[1].view(torch.int16))
