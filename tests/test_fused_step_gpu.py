"""The fused decode step (append + first cross-decoder layer in one launch) against
the separate calls and the oracle, for the bf16 and e4m3 caches."""
import numpy as np
import pytest
import torch

from tests.helpers import (ATOL, gpu_out, oracle_e4m3_pools, oracle_e4m3_step_out, oracle_pools,
                           oracle_step_out, pool_bits, oracle_bits)
from workloads import SMALL, page_scales, pure_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def N():
    from yoco_shared_kv_gb300 import build
    build.build()
    from yoco_shared_kv_gb300 import _native
    return _native


@pytest.fixture(scope="module")
def P(N):
    from yoco_shared_kv_gb300 import pipeline
    return pipeline


def _pair(P, wl, kv):
    sc = page_scales(wl) if kv == "e4m3" else None
    a = P.DeviceWorkload(wl, kv=kv, page_scales=sc)
    b = P.DeviceWorkload(wl, kv=kv, page_scales=sc)
    return a, b, sc


def _wide_decode():
    # 16 query heads per kv head at head_dim 256: two 8-head tiles, the queries in the
    # warp's shared-memory tile
    return pure_decode(8100, num_reqs=5, ctx_lo=1, ctx_hi=600, H_q=32, H_kv=2, D=256, bs=16,
                       layers=2)


@pytest.mark.parametrize("kv", ["native", "e4m3"])
@pytest.mark.parametrize("idx", [1, 4, "wide"])
def test_fused_step_equals_separate_calls(P, idx, kv):
    wl = _wide_decode() if idx == "wide" else SMALL[idx]()
    a, b, sc = _pair(P, wl, kv)
    for dw in (a, b):
        dw.run_fill()
    for i in range(len(wl.steps)):
        assert a.decode_only(i)
        a.run_step(i)      # append, select, every layer
        b.fused_step(i)    # append fused into layer 0, then every later layer
    torch.cuda.synchronize()
    assert a.error_bits() == 0 and b.error_bits() == 0
    assert torch.equal(a.k_cache.view(torch.uint8), b.k_cache.view(torch.uint8))
    assert torch.equal(a.v_cache.view(torch.uint8), b.v_cache.view(torch.uint8))
    for i in range(len(wl.steps)):
        # same kernel and the same key bits, so the same outputs bit for bit
        assert torch.equal(a.steps[i].out.view(torch.int16), b.steps[i].out.view(torch.int16))
    # and against the oracle (cache bit-exact, layer 0 and the last layer within tolerance)
    st = wl.steps[-1]
    if kv == "e4m3":
        kp, vp = oracle_e4m3_pools(wl, sc)
        assert np.array_equal(b.k_cache.cpu().numpy(), kp)
        ref = oracle_e4m3_step_out(wl, st, kp, vp, sc, layers=[0, wl.layers - 1])
    else:
        kp, vp = oracle_pools(wl)
        assert np.array_equal(pool_bits(b.k_cache), oracle_bits(kp))
        ref = oracle_step_out(wl, st, layers=[0, wl.layers - 1])
    got = gpu_out(b.steps[-1].out)[[0, wl.layers - 1]][:, :st.rows_upper]
    assert np.abs(got - ref).max() <= ATOL["bf16"]


def test_fused_step_flags_a_batch_that_is_not_decode(P, N):
    wl = SMALL[2]()  # mixed: prefill requests schedule many tokens
    dw = P.DeviceWorkload(wl)
    dw.run_fill()
    i = len(wl.steps) - 1
    assert not dw.decode_only(i)
    ds = dw.steps[i]
    d = ds.dev
    R = ds.num_reqs
    # feed the first R token rows as if they were the requests' single tokens
    N.yoco_cross_decode_step(d["q"][0][:R].contiguous(), d["k_new"][:R].contiguous(),
                             d["v_new"][:R].contiguous(), dw.k_cache, dw.v_cache, None,
                             torch.empty_like(d["q"][0][:R]), d["block_table"], d["seq_lens"],
                             d["qsl"], ds.max_seq_len, wl.scale, ds.workspace, dw.err)
    torch.cuda.synchronize()
    assert dw.error_bits() & N.DEVERR_OFFSETS
