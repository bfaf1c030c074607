"""The persisting L2 window over the shared-prefix pages, on the workload it
fits: the shared-prefix batch, whose 4096-token prefix is referenced by every
request's block table ("KV cache memory systems", "Prefix caching needs
identity rules") and re-read by every serial cross-decoder layer ("YOCO
论文与推理数据流详解" §11).

The window is a cache hint: with it set, every layer's output must be the
same bits as without it, and within tolerance of the oracle."""
import numpy as np
import pytest
import torch

from tests.helpers import ATOL, gpu_out, oracle_step_out
from workloads import FULL, SMALL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def PN():
    from yoco_shared_kv_gb300 import build
    build.build()
    from yoco_shared_kv_gb300 import _native, pipeline
    return pipeline, _native


def _prefix_span(wl, k_cache):
    """(base tensor view, bytes) of the K pool's physical pages that hold the prefix."""
    n_prefix_blocks = wl.prefix_len // wl.block_size
    pages = np.concatenate([np.asarray(p[:n_prefix_blocks]) for p in wl.req_pages])
    lo, hi = int(pages.min()), int(pages.max()) + 1
    page_bytes = k_cache[0].numel() * k_cache.element_size()
    return k_cache[lo], (hi - lo) * page_bytes


@pytest.mark.parametrize("size", ["small", "full"])
def test_l2_window_leaves_outputs_unchanged(PN, size):
    P, N = PN
    wl = (SMALL if size == "small" else FULL)[4]()
    dw = P.DeviceWorkload(wl)
    dw.run_fill()
    dw.run_step(0)  # no window: the reference outputs of every layer
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    ds = dw.steps[0]
    ref_bits = ds.out.clone()
    stream = torch.cuda.Stream()
    base, nbytes = _prefix_span(wl, dw.k_cache)
    N.yoco_set_l2_window(base, nbytes, -1.0, stream=stream)
    try:
        ds.out.fill_(float("nan"))
        with torch.cuda.stream(stream):
            for layer in range(wl.layers):
                dw.attend(ds, layer, stream=stream)
        stream.synchronize()
    finally:
        N.yoco_set_l2_window(None, 0, stream=stream)  # clear: window and set-aside
    assert dw.error_bits() == 0
    assert torch.equal(ds.out.view(torch.int16), ref_bits.view(torch.int16))
    got = gpu_out(ds.out)
    assert np.isfinite(got).all()
    step = wl.steps[0]
    if size == "small":
        ref = oracle_step_out(wl, step)
        assert np.abs(got - ref).max() <= ATOL["bf16"]
    else:
        n = step.rows_upper
        rng = np.random.default_rng(44)
        rows = sorted(set([0, n - 1] + rng.choice(n, size=3, replace=False).tolist()))
        layers = [0, wl.layers - 1]
        ref = oracle_step_out(wl, step, layers=layers, rows=rows)
        assert np.abs(got[layers][:, rows] - ref).max() <= ATOL["bf16"]
