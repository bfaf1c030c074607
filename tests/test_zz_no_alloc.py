"""The allocation-free attention entry point against the regular one.

yoco_cross_attn_paged_noalloc serves callers that cannot allocate device
memory (graph-capture regions, engines with a fixed memory budget, plugin
hosts without an allocator): it keeps its scratch in a fixed array inside
the library instead of a caller workspace. It must give the same result as
yoco_cross_attn_paged on the same inputs, call after call, since every call
shares (and overwrites) that array.

This file is named so pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests.helpers import ATOL, gpu_out, oracle_step_out
from workloads import SMALL

pytestmark = pytest.mark.gpu


def _abi():
    from yoco_shared_kv_gb300 import build
    build.build()
    from yoco_shared_kv_gb300 import _native
    return _native


def _call_noalloc(N, dw, ds, layer, out):
    """Straight through the C ABI (ctypes), no Python wrapper logic."""
    q = ds.dev["q"][layer]
    k = dw.k_cache
    num_blocks, H_kv, bs, D = k.shape
    rows, H_q, _ = q.shape
    bt = ds.dev["block_table"]
    st = N.lib.yoco_cross_attn_paged_noalloc(
        q.data_ptr(), k.data_ptr(), dw.v_cache.data_ptr(), out.data_ptr(), bt.data_ptr(),
        bt.shape[1], ds.dev["seq_lens"].data_ptr(), ds.cqsl.data_ptr(), ds.num_reqs, rows,
        ds.max_seq_len, H_q, H_kv, D, bs, num_blocks, ctypes.c_float(dw.wl.scale),
        N.dtype_code(q.dtype), dw.err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return st


@pytest.mark.parametrize("idx", [1, 3, 0])
def test_noalloc_matches_workspace_entry_point(idx):
    N = _abi()
    from yoco_shared_kv_gb300 import pipeline as P
    wl = SMALL[idx]()
    dw = P.DeviceWorkload(wl)
    dw.run_fill()
    i = len(wl.steps) - 1
    for j in range(i):
        dw.run_step(j)
    dw.run_step(i)  # regular entry point: every layer into ds.out
    ds = dw.steps[i]
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    need = N.yoco_cross_attn_workspace_size(ds.rows_upper, wl.num_q_heads, wl.num_kv_heads,
                                            wl.head_dim, wl.block_size, ds.max_seq_len,
                                            P.torch_dtype(wl.dtype))
    assert need <= N.yoco_cross_attn_noalloc_capacity()
    # the workspace entry with the flags the allocation-free entry uses (none):
    # the same kernels on the same inputs in the same order, so bit-identical
    refs = {}
    for layer in (0, wl.layers - 1):
        refs[layer] = torch.full_like(ds.out[layer], float("nan"))
        N.yoco_cross_attn_paged(ds.dev["q"][layer], dw.k_cache, dw.v_cache, refs[layer],
                                ds.dev["block_table"], ds.dev["seq_lens"], ds.cqsl,
                                ds.max_seq_len, wl.scale, ds.workspace, dw.err, flags=0)
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    oracle_ref = oracle_step_out(wl, wl.steps[i], layers=[0])[0]
    for call in range(2):  # two calls in a row share the one scratch array
        for layer in (0, wl.layers - 1):
            out = torch.full_like(ds.out[layer], float("nan"))
            assert _call_noalloc(N, dw, ds, layer, out) == N.YOCO_OK
            torch.cuda.synchronize()
            assert dw.error_bits() == 0
            got = gpu_out(out)
            assert np.isfinite(got).all()
            assert torch.equal(out, refs[layer]), (idx, call, layer)
            # and the regular pipeline (its own flags) within tolerance
            assert np.abs(got - gpu_out(ds.out[layer])).max() <= ATOL[wl.dtype]
            if layer == 0:  # one layer straight against the oracle
                assert np.abs(got - oracle_ref).max() <= ATOL[wl.dtype], (idx, call)


def test_noalloc_rejects_bounds_beyond_its_array():
    N = _abi()
    cap = N.yoco_cross_attn_noalloc_capacity()
    # the fp32 path's split grid, at the row count that makes it largest (16 heads,
    # head_dim 256, long contexts), needs more than the array holds
    H_q, H_kv, D, bs, ctx = 16, 2, 256, 16, 65536
    rows = max(range(1, 2048),
               key=lambda r: N.yoco_cross_attn_workspace_size(r, H_q, H_kv, D, bs, ctx,
                                                              torch.float32))
    need = N.yoco_cross_attn_workspace_size(rows, H_q, H_kv, D, bs, ctx, torch.float32)
    assert need > cap
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    st = N.lib.yoco_cross_attn_paged_noalloc(
        dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(),
        1, dummy.data_ptr(), dummy.data_ptr(), 1, rows, ctx, H_q, H_kv, D, bs, 1,
        ctypes.c_float(0.0625), N.YOCO_F32, None, None)
    assert st == N.YOCO_ERR_WORKSPACE  # rejected before any launch
