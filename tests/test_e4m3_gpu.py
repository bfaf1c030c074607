"""e4m3 cache on the GPU vs the oracle, through the C ABI: the quantising
append bit for bit (whole pools), attention over the dequantised cache within
the bf16 tolerance, bit-identical results under a page permutation, and the
scale-range flag."""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import ATOL, gpu_out, oracle_e4m3_pools, oracle_e4m3_step_out, oracle_step_out
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


def _run(P, wl, scales, layers=None, alternate="auto"):
    dw = P.DeviceWorkload(wl, kv="e4m3", page_scales=scales, alternate=alternate)
    dw.run_fill()
    for i in range(len(wl.steps)):
        dw.run_step(i, layers=layers)
    torch.cuda.synchronize()
    return dw


def _check_steps(wl, dw, scales, layers, rows=None):
    kp, vp = oracle_e4m3_pools(wl, scales)
    assert np.array_equal(dw.k_cache.cpu().numpy(), kp)
    assert np.array_equal(dw.v_cache.cpu().numpy(), vp)
    worst = 0.0
    for i, step in enumerate(wl.steps):
        ref = oracle_e4m3_step_out(wl, step, kp, vp, scales, layers=layers)
        got = gpu_out(dw.steps[i].out)[list(layers)][:, :step.rows_upper]
        assert np.isfinite(got).all()
        worst = max(worst, float(np.abs(got - ref).max()))
    assert worst <= ATOL["bf16"], worst
    return worst


@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_e4m3_step_matches_oracle(P, idx):
    wl = SMALL[idx]()
    scales = page_scales(wl)
    dw = _run(P, wl, scales)
    assert dw.error_bits() == 0
    _check_steps(wl, dw, scales, layers=[0, 1, wl.layers - 1])


@pytest.mark.parametrize("H_q,H_kv,D,bs", [(8, 2, 128, 16), (16, 1, 256, 32), (4, 4, 128, 32),
                                           (32, 2, 256, 16), (6, 3, 256, 16), (16, 1, 128, 16),
                                           (8, 2, 256, 32), (4, 1, 128, 32), (10, 2, 128, 32),
                                           (12, 1, 256, 16)])
def test_e4m3_shapes(P, H_q, H_kv, D, bs):
    wl = pure_decode(6000 + H_q * 7 + D, num_reqs=5, ctx_lo=1, ctx_hi=900, H_q=H_q, H_kv=H_kv,
                     D=D, bs=bs, layers=2)
    scales = page_scales(wl)
    dw = _run(P, wl, scales)
    assert dw.error_bits() == 0
    _check_steps(wl, dw, scales, layers=[0, 1])


def test_e4m3_block_edges_and_single_key(P):
    wl = pure_decode(6100, explicit_lens=[1, 16, 17, 32, 33, 2049], layers=2, D=128)
    scales = page_scales(wl)
    dw = _run(P, wl, scales)
    assert dw.error_bits() == 0
    _check_steps(wl, dw, scales, layers=[0, 1])
    # one key: the output is that key's dequantised value (one bf16 rounding away)
    kp, vp = oracle_e4m3_pools(wl, scales)
    st = wl.steps[0]
    V = oracle.e4m3_gather(vp, scales, 1, st.block_table[0], 1)[0]
    G = wl.num_q_heads // wl.num_kv_heads
    got = gpu_out(dw.steps[0].out)[0, 0]
    want = np.repeat(V, G, axis=0)
    assert np.abs(got - want).max() <= np.abs(want).max() * 2.0 ** -8


def test_e4m3_page_permutation_bit_identical(P):
    wl = SMALL[1]()
    scales = page_scales(wl)
    a = _run(P, wl, scales, alternate=False)
    out_a = a.steps[0].out.clone()
    # move every page (and its scale record) to another physical slot
    rng = np.random.default_rng(9)
    perm = rng.permutation(wl.num_blocks).astype(np.int32)
    for st in ([wl.fill] if wl.fill is not None else []) + wl.steps:
        st.block_table = np.where(st.block_table >= 0, perm[np.maximum(st.block_table, 0)],
                                  st.block_table).astype(np.int32)
    sc2 = np.zeros_like(scales)
    sc2[perm] = scales
    b = _run(P, wl, sc2, alternate=False)
    assert torch.equal(out_a.view(torch.int16), b.steps[0].out.view(torch.int16))


def test_e4m3_quantisation_error_vs_bf16_cache(P):
    """What the 8-bit cache costs in accuracy: its output against the oracle over
    the unquantised bf16 cache (reported by the assertion message)."""
    wl = SMALL[1]()
    scales = page_scales(wl)
    dw = _run(P, wl, scales)
    ref = oracle_step_out(wl, wl.steps[0], layers=[0])
    got = gpu_out(dw.steps[0].out)[[0]][:, :wl.steps[0].rows_upper]
    err = np.abs(got - ref)
    # e4m3 keeps 4 significant bits (half step 1/16 relative); on this workload the
    # output moved by 0.125 at most and 0.0071 on average when first measured
    print(f"e4m3 vs bf16 cache: max {err.max():.4f} mean {err.mean():.5f}")
    assert err.max() < 0.25 and err.mean() < 0.015, (err.max(), err.mean())


def test_e4m3_append_tie_and_bad_scale(P, N):
    """The float32-division tie case lands on the oracle's codes; a page with a
    zero scale is not written and flags YOCO_DEVERR_SCALE; attention over a page
    whose scale is out of range flags it too."""
    H_kv, D, bs = 1, 128, 16
    x = np.zeros((2, H_kv, D), dtype=np.float32)
    x[:, 0, :3] = [1.3671875, -1.3671875, 2.734375]
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    scales = np.zeros((4, H_kv, 4), np.float32)
    scales[..., 0], scales[..., 1] = 7.0, 3.5
    scales[3, 0, 0] = 0.0  # page 3 cannot be written
    bt = np.array([[1], [3]], np.int32)
    qsl, sl = np.array([0, 1, 2], np.int32), np.array([1, 1], np.int32)
    kp = np.full((4, H_kv, bs, D), 0xFF, np.uint8)
    vp = kp.copy()
    assert oracle.kv_append_e4m3(bits, bits, kp, vp, scales, bt, sl, qsl, bs) == 1
    dev = "cuda"
    kc = torch.full(kp.shape, 0xFF, dtype=torch.uint8, device=dev)
    vc = kc.clone()
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kn = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)
    N.yoco_kv_append_e4m3(kn, kn, kc, vc, torch.from_numpy(scales).to(dev),
                          torch.from_numpy(bt).to(dev), torch.from_numpy(sl).to(dev),
                          torch.from_numpy(qsl).to(dev), err)
    torch.cuda.synchronize()
    assert int(err.item()) == N.DEVERR_SCALE
    assert np.array_equal(kc.cpu().numpy(), kp) and np.array_equal(vc.cpu().numpy(), vp)
    # attention over page 1 with a V scale above 2^7: flagged
    sc_bad = scales.copy()
    sc_bad[1, 0, 1] = 1000.0
    q = torch.zeros((1, 1, D), dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(q)
    ws = torch.empty(N.yoco_cross_attn_workspace_size(1, 1, 1, D, bs, 1, torch.float8_e4m3fn),
                     dtype=torch.uint8, device=dev)
    err.zero_()
    N.yoco_cross_attn_paged_e4m3(q, kc, vc, torch.from_numpy(sc_bad).to(dev), out,
                                 torch.from_numpy(bt[:1]).to(dev), torch.from_numpy(sl[:1]).to(dev),
                                 torch.tensor([0, 1], dtype=torch.int32, device=dev), 1,
                                 D ** -0.5, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) & N.DEVERR_SCALE


def test_e4m3_empty_row_and_bad_page_flagged(P, N):
    wl = SMALL[1]()
    scales = page_scales(wl)
    dw = _run(P, wl, scales)
    ds = dw.steps[0]
    d = ds.dev
    sc = dw.page_scales
    # seq_len 0 for request 0: its row has no key -> zero output + flag
    sl = d["seq_lens"].clone()
    sl[0] = 0
    out = torch.full_like(ds.out[0], 3.0)
    dw.err.zero_()
    N.yoco_cross_attn_paged_e4m3(d["q"][0], dw.k_cache, dw.v_cache, sc, out, d["block_table"], sl,
                                 ds.cqsl, ds.max_seq_len, wl.scale, ds.workspace, dw.err)
    torch.cuda.synchronize()
    assert dw.error_bits() & N.DEVERR_EMPTY_ROW
    assert (out[0] == 0).all()
    # a page id past the pool: flagged, skipped, no fault
    bt = d["block_table"].clone()
    bt[3, 2] = -4
    dw.err.zero_()
    N.yoco_cross_attn_paged_e4m3(d["q"][0], dw.k_cache, dw.v_cache, sc, out, bt, d["seq_lens"],
                                 ds.cqsl, ds.max_seq_len, wl.scale, ds.workspace, dw.err)
    torch.cuda.synchronize()
    assert dw.error_bits() & N.DEVERR_PAGE_RANGE


@pytest.mark.parametrize("kv", ["native", "e4m3"])
def test_fused_step_bad_page_flagged(P, N, kv):
    wl = SMALL[1]()
    sc = page_scales(wl) if kv == "e4m3" else None
    dw = P.DeviceWorkload(wl, kv=kv, page_scales=sc)
    dw.run_fill()
    ds = dw.steps[0]
    d = ds.dev
    bt = d["block_table"].clone()
    r = 2
    last_page = (int(wl.steps[0].seq_lens[r]) - 1) // wl.block_size
    bt[r, last_page] = wl.num_blocks + 5  # the new token's page is out of the pool
    before = dw.k_cache.clone()
    N.yoco_cross_decode_step(d["q"][0], d["k_new"], d["v_new"], dw.k_cache, dw.v_cache,
                             dw.page_scales, ds.out[0], bt, d["seq_lens"], d["qsl"],
                             ds.max_seq_len, wl.scale, ds.workspace, dw.err)
    torch.cuda.synchronize()
    assert dw.error_bits() & N.DEVERR_PAGE_RANGE
    # nothing was written for the skipped token; the other requests' tokens were
    changed = (dw.k_cache.view(torch.uint8) != before.view(torch.uint8))
    assert changed.any()


@pytest.mark.parametrize("H_q,H_kv,D,bs,draft", [(8, 2, 256, 16, 4), (4, 2, 128, 32, 3),
                                                 (4, 4, 128, 16, 10), (16, 2, 256, 32, 2)])
def test_e4m3_row_groups(P, H_q, H_kv, D, bs, draft):
    """Several cross rows per request over the e4m3 cache: rows grouped on one walk
    (8- and 16-wide groups; the second layer walks its pages backwards)."""
    from workloads import spec_decode
    wl = spec_decode(7400 + H_q + draft, num_reqs=5, ctx_lo=1, ctx_hi=700, draft=draft, H_q=H_q,
                     H_kv=H_kv, D=D, bs=bs, layers=2)
    scales = page_scales(wl)
    dw = _run(P, wl, scales, alternate=True)
    assert dw.error_bits() == 0
    _check_steps(wl, dw, scales, layers=[0, 1])
