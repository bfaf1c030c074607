"""GPU path vs the CPU oracle, element by element (bit-exact for append and
selection; max-abs tolerance for attention), through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import (ATOL, gpu_out, oracle_bits, oracle_pools, oracle_step_out, pool_bits)
from workloads import SMALL, Workload, pure_decode

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


def _i32(x):
    return torch.tensor(np.asarray(x, dtype=np.int32), device="cuda")


# ------------------------------------------------------------------ selection


def _gpu_select(N, qsl, rpr=None, cap=None):
    qsl = np.asarray(qsl, dtype=np.int32)
    R = len(qsl) - 1
    cap = cap or max(int(qsl[-1]) if R else 0, 1) + 64
    rows = torch.full((cap,), -7, dtype=torch.int32, device="cuda")
    cq = torch.full((R + 1,), -7, dtype=torch.int32, device="cuda")
    nr = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    N.yoco_select_cross_rows(_i32(qsl), None if rpr is None else _i32(rpr), rows, cq, nr, err)
    torch.cuda.synchronize()
    n = int(nr.item())
    return rows.cpu().numpy(), cq.cpu().numpy(), n, int(err.item())


def test_select_worked_example(N, golden_dir):
    import json, os
    g = json.load(open(os.path.join(golden_dir, "select_vllm_example.json")))
    rows, cq, n, err = _gpu_select(N, g["query_start_loc"], g["rows_per_req"])
    assert err == 0 and n == 4
    assert rows[:n].tolist() == g["expected_rows"]
    assert cq.tolist() == g["expected_cross_query_start_loc"]
    assert (rows[n:] == -7).all()  # nothing written past the rows


@pytest.mark.parametrize("seed", range(12))
def test_select_random_bit_exact(N, seed):
    rng = np.random.default_rng(100 + seed)
    R = int(rng.choice([1, 7, 33, 1023, 1024, 1025, 3000, 5000]))
    qlen = rng.integers(0, 12, size=R)
    qlen[rng.random(R) < 0.6] = 1
    qsl = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    rpr = None if seed % 3 == 0 else rng.integers(0, 6, size=R).astype(np.int32)
    rows, cq, n, err = _gpu_select(N, qsl, rpr)
    o_rows, o_cq, o_n = oracle.select_cross_rows(qsl, rpr)
    assert err == 0 and n == o_n
    assert np.array_equal(rows[:n], o_rows)
    assert np.array_equal(cq, o_cq)


def test_select_edge_cases(N):
    rows, cq, n, err = _gpu_select(N, [0])
    assert n == 0 and cq.tolist() == [0] and err == 0
    rows, cq, n, err = _gpu_select(N, [0, 0, 3, 3])
    assert n == 1 and rows[0] == 2 and cq.tolist() == [0, 0, 1, 1]
    rows, cq, n, err = _gpu_select(N, [0, 2, 5], [7, 0])
    assert n == 2 and rows[:2].tolist() == [0, 1] and cq.tolist() == [0, 2, 2]
    _, _, _, err = _gpu_select(N, [0, 3, 2])
    assert err & N.DEVERR_OFFSETS


# --------------------------------------------------------------------- append


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_append_bit_exact_whole_pool(P, idx):
    wl = SMALL[idx]()
    dw = P.DeviceWorkload(wl)
    dw.run_fill()
    for i in range(len(dw.steps)):
        dw.append(dw.steps[i])
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    kp, vp = oracle_pools(wl)
    assert np.array_equal(pool_bits(dw.k_cache), oracle_bits(kp))
    assert np.array_equal(pool_bits(dw.v_cache), oracle_bits(vp))


def test_append_bad_page_sets_error_and_skips(P, N):
    wl = SMALL[1]()
    dw = P.DeviceWorkload(wl)
    ds = dw.steps[0]
    bt = ds.dev["block_table"].clone()
    bt[0, :] = wl.num_blocks + 5  # request 0 points past the pool
    N.yoco_kv_append(ds.dev["k_new"], ds.dev["v_new"], dw.k_cache, dw.v_cache, bt,
                     ds.dev["seq_lens"], ds.dev["qsl"], dw.err)
    torch.cuda.synchronize()
    assert dw.error_bits() & N.DEVERR_PAGE_RANGE
    # everything else was still written, exactly as the oracle skips it
    step = wl.steps[0]
    kp, vp = wl.empty_pool(), wl.empty_pool()
    bad_bt = step.block_table.copy()
    bad_bt[0, :] = wl.num_blocks + 5
    skipped = oracle.kv_append(step.k_new, step.v_new, kp, vp, bad_bt, step.seq_lens,
                               step.query_start_loc, wl.block_size)
    assert skipped == wl.num_kv_heads
    assert np.array_equal(pool_bits(dw.k_cache), oracle_bits(kp))


# ------------------------------------------------------------------ attention


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_step_matches_oracle(P, idx):
    """Fill + every step (append -> select -> all layers) vs the oracle, every output."""
    wl = SMALL[idx]()
    dw = P.DeviceWorkload(wl)
    dw.run_fill()
    for i, step in enumerate(wl.steps):
        dw.run_step(i)
        torch.cuda.synchronize()
        assert dw.error_bits() == 0
        ds = dw.steps[i]
        o_rows, o_cq, n = oracle.select_cross_rows(step.query_start_loc, step.rows_per_req)
        assert int(ds.num_rows.item()) == n
        assert np.array_equal(ds.row_indices.cpu().numpy()[:n], o_rows)
        assert np.array_equal(ds.cqsl.cpu().numpy(), o_cq)
        ref = oracle_step_out(wl, step)
        got = gpu_out(ds.out)
        assert np.isfinite(got).all()
        err = np.abs(got - ref).max()
        assert err <= ATOL[wl.dtype], (wl.name, i, err)


def test_attention_page_permutation_bit_identical(P):
    a = SMALL[1]()
    b = SMALL[1]()
    perm = np.random.default_rng(11).permutation(b.num_blocks).astype(np.int32)
    for st in [b.fill] + b.steps:
        st.block_table = perm[st.block_table]
    outs = []
    for wl in (a, b):
        dw = P.DeviceWorkload(wl)
        dw.run_all()
        torch.cuda.synchronize()
        assert dw.error_bits() == 0
        outs.append(dw.steps[0].out.cpu())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_attention_single_key_and_block_edges(P):
    """Contexts of 1, block_size, block_size + 1 tokens (and a long one) in one batch."""
    wl = pure_decode(3001, explicit_lens=[1, 16, 17, 32, 33, 2049], layers=2)
    dw = P.DeviceWorkload(wl)
    dw.run_all()
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    got = gpu_out(dw.steps[0].out)
    ref = oracle_step_out(wl, wl.steps[0])
    assert np.abs(got - ref).max() <= ATOL["bf16"]
    # a single key returns V exactly (bf16 rounding of an exactly representable value)
    K, V = wl.request_kv(0)
    v0 = oracle.widen(V[0], "bf16")  # [H_kv, D]
    G = wl.num_q_heads // wl.num_kv_heads
    for h in range(wl.num_q_heads):
        assert np.array_equal(got[0, 0, h], v0[h // G])


@pytest.mark.parametrize("H_q,H_kv,D,bs", [(4, 4, 64, 16), (6, 2, 128, 32), (12, 1, 64, 32),
                                           (16, 2, 256, 16), (2, 1, 128, 16), (16, 16, 128, 32),
                                           (16, 1, 256, 32), (32, 2, 256, 16), (8, 1, 64, 16),
                                           (10, 2, 128, 16), (7, 1, 256, 32)])
def test_attention_shapes(P, H_q, H_kv, D, bs):
    wl = pure_decode(4000 + H_q * 7 + D, num_reqs=5, ctx_lo=1, ctx_hi=900, H_q=H_q, H_kv=H_kv,
                     D=D, bs=bs, layers=2)
    dw = P.DeviceWorkload(wl)
    dw.run_all()
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    got = gpu_out(dw.steps[0].out)
    ref = oracle_step_out(wl, wl.steps[0])
    assert np.abs(got - ref).max() <= ATOL["bf16"]


def test_attention_fewer_pages_than_workers(P):
    """A batch of a few short rows: most CTAs and warps of the persistent grid get no page."""
    for lens in ([5], [1, 3], [40, 1, 17]):
        wl = pure_decode(3100 + len(lens), explicit_lens=lens, layers=2)
        dw = P.DeviceWorkload(wl)
        dw.run_all()
        torch.cuda.synchronize()
        assert dw.error_bits() == 0
        got = gpu_out(dw.steps[0].out)
        ref = oracle_step_out(wl, wl.steps[0])
        assert np.abs(got - ref).max() <= ATOL["bf16"], lens


def test_attention_one_long_row_many_ctas(P):
    """One row far longer than a CTA slice: its pieces are merged across many CTAs."""
    wl = pure_decode(3200, explicit_lens=[60000], H_q=16, H_kv=1, D=128, bs=32, layers=2)
    dw = P.DeviceWorkload(wl)
    dw.run_all()
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    got = gpu_out(dw.steps[0].out)
    ref = oracle_step_out(wl, wl.steps[0])
    assert np.abs(got - ref).max() <= ATOL["bf16"]


@pytest.mark.parametrize("D", [64, 128, 256])
def test_attention_fp32_shapes(P, D):
    wl = pure_decode(5000 + D, num_reqs=4, ctx_lo=1, ctx_hi=700, H_q=8, H_kv=2, D=D, bs=16,
                     layers=2, dtype="f32")
    dw = P.DeviceWorkload(wl)
    dw.run_all()
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    got = gpu_out(dw.steps[0].out)
    ref = oracle_step_out(wl, wl.steps[0])
    assert np.abs(got - ref).max() <= ATOL["f32"]


def test_multi_row_requests_bottom_right_causal(P):
    """rows_per_req > 1: trailing rows of a prefill see their own causal prefix."""
    from workloads import mixed_step
    wl = mixed_step(6001, n_decode=3, dec_lo=50, dec_hi=300, n_prefill=3, pre_lo=20, pre_hi=200,
                    layers=2, rows_per_req=[1, 1, 1, 4, 2, 7])
    dw = P.DeviceWorkload(wl)
    dw.run_all()
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    got = gpu_out(dw.steps[0].out)
    ref = oracle_step_out(wl, wl.steps[0])
    assert np.abs(got - ref).max() <= ATOL["bf16"]


def test_attention_empty_row_and_bad_page_flagged(P, N):
    wl = SMALL[1]()
    dw = P.DeviceWorkload(wl)
    dw.run_all()
    ds = dw.steps[0]
    # seq_len 0 for request 0: its row has no key -> zero output + flag
    sl = ds.dev["seq_lens"].clone()
    sl[0] = 0
    out = torch.full_like(ds.out[0], 3.0)
    dw.err.zero_()
    N.yoco_cross_attn_paged(ds.dev["q"][0], dw.k_cache, dw.v_cache, out, ds.dev["block_table"],
                            sl, ds.cqsl, ds.max_seq_len, wl.scale, ds.workspace, dw.err)
    torch.cuda.synchronize()
    assert dw.error_bits() & N.DEVERR_EMPTY_ROW
    assert (out[0] == 0).all()
    # a page id past the pool: flagged, skipped, no fault
    bt = ds.dev["block_table"].clone()
    bt[3, 2] = -4
    dw.err.zero_()
    N.yoco_cross_attn_paged(ds.dev["q"][0], dw.k_cache, dw.v_cache, out, bt, ds.dev["seq_lens"],
                            ds.cqsl, ds.max_seq_len, wl.scale, ds.workspace, dw.err)
    torch.cuda.synchronize()
    assert dw.error_bits() & N.DEVERR_PAGE_RANGE


def test_workspace_too_small_is_rejected(P, N):
    wl = SMALL[3]()
    dw = P.DeviceWorkload(wl)
    ds = dw.steps[0]
    with pytest.raises(N.YocoError) as e:
        N.yoco_cross_attn_paged(ds.dev["q"][0], dw.k_cache, dw.v_cache, ds.out[0],
                                ds.dev["block_table"], ds.dev["seq_lens"], ds.cqsl, 131072,
                                wl.scale, ds.workspace[:16], dw.err)
    assert e.value.status == N.YOCO_ERR_WORKSPACE


@pytest.mark.parametrize("lens,H_q,H_kv,D,bs", [([5], 8, 2, 256, 16), ([1, 3, 300], 8, 2, 128, 32),
                                               ([40, 1, 17, 2000], 16, 1, 128, 32),
                                               ([60000], 16, 1, 128, 32)])
def test_attention_writes_only_its_outputs(P, N, lens, H_q, H_kv, D, bs):
    """Canary regions around `out` stay untouched; scratch starts as NaN bytes."""
    wl = pure_decode(3300 + len(lens), explicit_lens=lens, H_q=H_q, H_kv=H_kv, D=D, bs=bs,
                     layers=1)
    dw = P.DeviceWorkload(wl)
    dw.run_fill()
    dw.run_step(0)
    torch.cuda.synchronize()
    ds = dw.steps[0]
    n_out = ds.out[0].numel()
    pad = 4096
    big = torch.full((pad + n_out + pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = big[pad:pad + n_out].view(ds.out[0].shape)
    ds.workspace.fill_(255)
    dw.plan(ds)  # the step's plan, then every other scratch byte is still NaN
    dw.attend(ds, 0, out=out)
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    assert (big[:pad] == 7.0).all() and (big[pad + n_out:] == 7.0).all()
    ref = oracle_step_out(wl, wl.steps[0])
    got = gpu_out(out)[None]
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= ATOL["bf16"]


def test_bounded_wait_gives_up_with_a_status(P, N):
    """A copy that never lands ends in YOCO_DEVERR_TIMEOUT, and the context stays usable."""
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    N.yoco_selftest_wait_timeout(err, 20000)  # 20 ms limit
    torch.cuda.synchronize()
    assert int(err.item()) & N.DEVERR_TIMEOUT
    # the same process keeps working: a normal step still matches the oracle
    wl = SMALL[1]()
    dw = P.DeviceWorkload(wl)
    dw.run_all()
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    got = gpu_out(dw.steps[0].out)
    ref = oracle_step_out(wl, wl.steps[0])
    assert np.abs(got - ref).max() <= ATOL["bf16"]


def test_chunked_prefill_and_speculative_rows(P):
    """Three steps: a prompt prefilled in chunks (no cross row until the last chunk),
    a decode, and a 3-token speculative verify asking for all trailing rows."""
    from workloads import chunked_prefill_spec
    wl = chunked_prefill_spec()
    dw = P.DeviceWorkload(wl)
    dw.run_fill()
    for i, step in enumerate(wl.steps):
        dw.run_step(i)
        torch.cuda.synchronize()
        assert dw.error_bits() == 0
        ds = dw.steps[i]
        o_rows, o_cq, n = oracle.select_cross_rows(step.query_start_loc, step.rows_per_req)
        assert int(ds.num_rows.item()) == n == step.rows_upper
        assert np.array_equal(ds.row_indices.cpu().numpy()[:n], o_rows)
        assert np.array_equal(ds.cqsl.cpu().numpy(), o_cq)
        got = gpu_out(ds.out)
        ref = oracle_step_out(wl, step)
        assert np.abs(got - ref).max() <= ATOL["bf16"], i
    kp, vp = oracle_pools(wl)
    assert np.array_equal(pool_bits(dw.k_cache), oracle_bits(kp))


@pytest.mark.parametrize("max_seq_len", [300, 1000])
def test_fp32_rows_beyond_max_seq_len_are_cut_and_flagged(P, N, max_seq_len):
    """fp32 split-KV path: a seq_len above the caller's max_seq_len bound.

    The split plan and its workspace are sized for max_seq_len keys per row
    (none at all when one split suffices), so the kernels cut such a row to
    its first max_seq_len keys and set POS_RANGE; nothing outside `out` and
    the workspace is written (canaries on both sides of each)."""
    import dataclasses
    lens = [150, 2000, 3000, 40]
    wl = pure_decode(3400 + max_seq_len, explicit_lens=lens, H_q=8, H_kv=2, D=128, bs=16,
                     layers=1, dtype="f32")
    dw = P.DeviceWorkload(wl)
    dw.run_fill()
    dw.run_step(0)  # append + select (+ layer 0 with the true bound)
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    ds = dw.steps[0]
    need = N.yoco_cross_attn_workspace_size(ds.rows_upper, wl.num_q_heads, wl.num_kv_heads,
                                            wl.head_dim, wl.block_size, max_seq_len,
                                            torch.float32)
    pad = 4096
    wsb = torch.full((pad + max(need, 16) + pad,), 0x5A, dtype=torch.uint8, device="cuda")
    ws = wsb[pad:pad + need] if need > 0 else None
    n_out = ds.out[0].numel()
    big = torch.full((pad + n_out + pad,), 7.0, dtype=torch.float32, device="cuda")
    out = big[pad:pad + n_out].view(ds.out[0].shape)
    dw.err.zero_()
    N.yoco_cross_attn_paged(ds.dev["q"][0], dw.k_cache, dw.v_cache, out, ds.dev["block_table"],
                            ds.dev["seq_lens"], ds.cqsl, max_seq_len, wl.scale, ws, dw.err)
    torch.cuda.synchronize()
    assert dw.error_bits() == N.DEVERR_POS_RANGE
    assert (big[:pad] == 7.0).all() and (big[pad + n_out:] == 7.0).all()
    assert (wsb[:pad] == 0x5A).all() and (wsb[pad + need:] == 0x5A).all()
    got = gpu_out(out)[None]
    assert np.isfinite(got).all()
    cut = dataclasses.replace(wl.steps[0], seq_lens=np.minimum(wl.steps[0].seq_lens, max_seq_len))
    ref = oracle_step_out(wl, cut)
    assert np.abs(got - ref).max() <= ATOL["f32"]


def _pair_workload(kind):
    """Workloads whose walks run on warp pairs (two 8-head tiles at head_dim 256)."""
    from workloads import spec_decode
    if kind == "wide":  # 16 query heads per kv head
        return pure_decode(8200, num_reqs=5, ctx_lo=1, ctx_hi=700, H_q=32, H_kv=2, D=256, bs=16,
                           layers=2)
    # four rows of a request at four heads per kv head: 16-wide row groups
    return spec_decode(8300, num_reqs=5, ctx_lo=1, ctx_hi=700, draft=4, layers=2)


def _workload(idx):
    return _pair_workload(idx) if isinstance(idx, str) else SMALL[idx]()


@pytest.mark.parametrize("idx", [1, 2, 3, 4, "wide", "spec"])
def test_planned_layers_equal_unplanned_calls(P, N, idx):
    """A layer reusing the step's plan (YOCO_ATTN_PLANNED) gives the same bits as
    a self-contained call that makes its own plan first, for both page walks (also
    on the warp-pair kernels)."""
    wl = _workload(idx)
    dw = P.DeviceWorkload(wl, alternate=True)
    dw.run_all()
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    ds = dw.steps[-1]
    for layer in range(wl.layers):
        flags = N.YOCO_ATTN_KEEP_TAIL | (N.YOCO_ATTN_REVERSE if layer % 2 else 0)
        out = torch.full_like(ds.out[layer], float("nan"))
        N.yoco_cross_attn_paged(ds.dev["q"][layer], dw.k_cache, dw.v_cache, out,
                                ds.dev["block_table"], ds.dev["seq_lens"], ds.cqsl,
                                ds.max_seq_len, wl.scale, ds.workspace, dw.err, flags=flags)
        torch.cuda.synchronize()
        assert dw.error_bits() == 0
        assert torch.equal(out.view(torch.int16), ds.out[layer].view(torch.int16)), layer
    ref = oracle_step_out(wl, wl.steps[-1])
    assert np.abs(gpu_out(ds.out) - ref).max() <= ATOL["bf16"]


@pytest.mark.parametrize("idx", [1, "wide", "spec"])
def test_planned_call_without_a_matching_plan_is_refused(P, N, idx):
    """YOCO_ATTN_PLANNED on a workspace that holds no plan, or a plan made for
    other shapes: the launch writes nothing and sets YOCO_DEVERR_PLAN (one warp per
    ring, and warp pairs: both warps of a pair leave together)."""
    wl = _workload(idx)
    dw = P.DeviceWorkload(wl)
    dw.run_all()
    torch.cuda.synchronize()
    ds = dw.steps[0]
    q = ds.dev["q"][0]
    args = (dw.k_cache, dw.v_cache)
    # no plan at all (scratch bytes all ones)
    ds.workspace.fill_(255)
    out = torch.full_like(ds.out[0], 5.0)
    dw.err.zero_()
    N.yoco_cross_attn_paged(q, *args, out, ds.dev["block_table"], ds.dev["seq_lens"], ds.cqsl,
                            ds.max_seq_len, wl.scale, ds.workspace, dw.err,
                            flags=N.YOCO_ATTN_PLANNED)
    torch.cuda.synchronize()
    assert dw.error_bits() == N.DEVERR_PLAN
    assert (out == 5.0).all()
    # a plan made for fewer rows than the call asks for
    rows = q.shape[0]
    N.yoco_cross_attn_plan(ds.dev["block_table"], ds.dev["seq_lens"], ds.cqsl, ds.max_seq_len,
                           rows - 1, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size,
                           dw.k_cache.shape[0], torch.bfloat16, ds.workspace, dw.err)
    dw.err.zero_()
    N.yoco_cross_attn_paged(q, *args, out, ds.dev["block_table"], ds.dev["seq_lens"], ds.cqsl,
                            ds.max_seq_len, wl.scale, ds.workspace, dw.err,
                            flags=N.YOCO_ATTN_PLANNED)
    torch.cuda.synchronize()
    assert dw.error_bits() == N.DEVERR_PLAN
    assert (out == 5.0).all()
    # the matching plan: accepted, and the result is the step's
    dw.plan(ds)
    dw.err.zero_()
    N.yoco_cross_attn_paged(q, *args, out, ds.dev["block_table"], ds.dev["seq_lens"], ds.cqsl,
                            ds.max_seq_len, wl.scale, ds.workspace, dw.err,
                            flags=N.YOCO_ATTN_PLANNED)
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    ref = oracle_step_out(wl, wl.steps[0], layers=[0])[0]
    assert np.abs(gpu_out(out) - ref).max() <= ATOL["bf16"]


def test_plan_is_reused_across_layers_and_replaced_per_step(P):
    """The chunked-prefill / speculative schedule: three steps with different
    metadata, each planned once and attended by every layer."""
    from workloads import chunked_prefill_spec
    wl = chunked_prefill_spec()
    dw = P.DeviceWorkload(wl)
    dw.run_fill()
    for i, step in enumerate(wl.steps):
        dw.run_step(i)
        torch.cuda.synchronize()
        assert dw.error_bits() == 0
        n = int(dw.steps[i].num_rows.item())
        got = gpu_out(dw.steps[i].out[:, :n])
        ref = oracle_step_out(wl, step)
        assert np.abs(got - ref).max() <= ATOL["bf16"], i


def test_speculative_rows_small_against_oracle(P):
    """Speculative verification: every request asks for its 4 trailing rows, each
    with its own bottom-right causal length (all rows, every layer)."""
    from workloads import MULTI_ROW_SMALL
    wl = MULTI_ROW_SMALL()
    dw = P.DeviceWorkload(wl)
    dw.run_all()
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    ref = oracle_step_out(wl, wl.steps[0])
    assert np.abs(gpu_out(dw.steps[0].out) - ref).max() <= ATOL["bf16"]


@pytest.mark.parametrize("H_q,H_kv,D,bs,draft", [(8, 2, 256, 16, 4), (4, 4, 128, 32, 3),
                                                 (2, 2, 64, 16, 7), (3, 1, 128, 16, 5),
                                                 (16, 1, 128, 32, 2), (8, 1, 128, 16, 2),
                                                 (2, 2, 64, 32, 12), (4, 2, 256, 32, 6),
                                                 (8, 2, 256, 16, 2)])
def test_row_groups_against_oracle_and_page_permutation(P, H_q, H_kv, D, bs, draft):
    """Several cross rows per request (max_rows above num_reqs): rows of a request
    share one walk over its pages in groups whose heads fill one 8-wide tile (8 / G
    rows, when the rows per request fit) or two (16 / G rows), each row with its own
    causal end. The cases cover both widths, the query tile in shared memory (head_dim
    256, two tiles) and a group of 16 one-head rows. Every row of every layer against
    the oracle, and bit-identical under a re-permutation of the physical pages."""
    from workloads import spec_decode
    seed = 7100 + H_q * 13 + D + draft
    a = spec_decode(seed, num_reqs=5, ctx_lo=1, ctx_hi=700, draft=draft, H_q=H_q, H_kv=H_kv,
                    D=D, bs=bs, layers=2)
    b = spec_decode(seed, num_reqs=5, ctx_lo=1, ctx_hi=700, draft=draft, H_q=H_q, H_kv=H_kv,
                    D=D, bs=bs, layers=2)
    perm = np.random.default_rng(seed).permutation(b.num_blocks).astype(np.int32)
    for st in [b.fill] + b.steps:
        st.block_table = perm[st.block_table]
    outs = []
    for wl in (a, b):
        dw = P.DeviceWorkload(wl, alternate=True)  # odd layers walk backwards
        dw.run_all()
        torch.cuda.synchronize()
        assert dw.error_bits() == 0
        outs.append(dw.steps[0].out.cpu())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    ref = oracle_step_out(a, a.steps[0])
    assert np.abs(outs[0].float().numpy().astype(np.float64) - ref).max() <= ATOL["bf16"]


def test_grouped_and_single_row_walks_agree(P, N):
    """The same speculative batch with max_rows = num_reqs + its rows (rows grouped on
    one walk) and, with the rows spread one per request (no grouping): both within
    tolerance of the oracle."""
    from workloads import spec_decode
    wl = spec_decode(7300, num_reqs=4, ctx_lo=30, ctx_hi=500, draft=4, layers=1)
    dw = P.DeviceWorkload(wl)
    dw.run_all()
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    ref = oracle_step_out(wl, wl.steps[0])[0]
    assert np.abs(gpu_out(dw.steps[0].out[0]) - ref).max() <= ATOL["bf16"]
    # one row per request: request r's four rows become four one-row requests with the
    # same pages and causal ends (seq_len - 3 .. seq_len), so max_rows == num_reqs
    st = wl.steps[0]
    ds = dw.steps[0]
    R = st.num_reqs
    bt = np.repeat(np.asarray(st.block_table), 4, axis=0)
    sl = np.concatenate([np.asarray(st.seq_lens)[r] - 3 + np.arange(4) for r in range(R)])
    cq = np.arange(4 * R + 1)
    out = torch.full_like(ds.out[0], float("nan"))
    N.yoco_cross_attn_paged(ds.dev["q"][0], dw.k_cache, dw.v_cache, out, _i32(bt),
                            _i32(sl.astype(np.int32)), _i32(cq), ds.max_seq_len, wl.scale,
                            ds.workspace, dw.err)
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    assert np.abs(gpu_out(out) - ref).max() <= ATOL["bf16"]


def test_row_group_with_an_empty_row(P, N):
    """A request whose seq_len is below its row count: its first row has no key and
    shares a group with rows that have keys. That row is zero-filled and flagged
    EMPTY_ROW; the others match the oracle's rows with keys."""
    from workloads import spec_decode
    wl = spec_decode(7500, num_reqs=3, ctx_lo=20, ctx_hi=200, draft=4, layers=1)
    dw = P.DeviceWorkload(wl)
    dw.run_all()
    torch.cuda.synchronize()
    ds = dw.steps[0]
    sl = ds.dev["seq_lens"].clone()
    sl[1] = 3  # request 1 has 4 rows: keys 0, 1, 2, 3 -> its first row has none
    out = torch.full_like(ds.out[0], 5.0)
    dw.err.zero_()
    N.yoco_cross_attn_paged(ds.dev["q"][0], dw.k_cache, dw.v_cache, out, ds.dev["block_table"],
                            sl, ds.cqsl, ds.max_seq_len, wl.scale, ds.workspace, dw.err)
    torch.cuda.synchronize()
    assert dw.error_bits() == N.DEVERR_EMPTY_ROW
    got = gpu_out(out)
    assert (got[4] == 0).all()  # request 1's first row
    assert np.isfinite(got).all()
    import dataclasses
    st = dataclasses.replace(wl.steps[0], seq_lens=sl.cpu().numpy())
    ref = oracle_step_out(wl, st, layers=[0], rows=[r for r in range(12) if r != 4])[0]
    assert np.abs(np.delete(got, 4, axis=0) - ref).max() <= ATOL["bf16"]


@pytest.mark.parametrize("kv", ["native", "e4m3"])
def test_loose_max_rows_over_one_row_requests(P, N, kv):
    """max_rows well above the rows the selection produced (a caller's loose bound): the
    launch then takes the 16-wide row-group kernel (max_rows / num_reqs = 4 rows per
    request at four heads per kv head) although every request has one row. The real rows
    match the oracle; rows past them are neither read nor written."""
    from workloads import page_scales
    wl = pure_decode(7600, num_reqs=6, ctx_lo=1, ctx_hi=800, layers=1)
    e4m3 = kv == "e4m3"
    dw = P.DeviceWorkload(wl, kv="e4m3", page_scales=page_scales(wl)) if e4m3 \
        else P.DeviceWorkload(wl)
    dw.run_all()
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    ds = dw.steps[0]
    R = ds.out.shape[1]
    cap = 4 * R
    q = torch.full((cap, wl.num_q_heads, wl.head_dim), float("nan"), dtype=torch.bfloat16,
                   device="cuda")
    q[:R] = ds.dev["q"][0]
    out = torch.full_like(q, 7.0)
    if e4m3:
        N.yoco_cross_attn_paged_e4m3(q, dw.k_cache, dw.v_cache, dw.page_scales, out,
                                     ds.dev["block_table"], ds.dev["seq_lens"], ds.cqsl,
                                     ds.max_seq_len, wl.scale, ds.workspace, dw.err)
    else:
        N.yoco_cross_attn_paged(q, dw.k_cache, dw.v_cache, out, ds.dev["block_table"],
                                ds.dev["seq_lens"], ds.cqsl, ds.max_seq_len, wl.scale,
                                ds.workspace, dw.err)
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    assert (out[R:] == 7.0).all()
    # the same rows as the step's own (exact max_rows) launch, and the oracle's
    assert np.abs(gpu_out(out[:R]) - gpu_out(ds.out[0])).max() <= ATOL["bf16"]
    if not e4m3:
        ref = oracle_step_out(wl, wl.steps[0])[0]
        assert np.abs(gpu_out(out[:R]) - ref).max() <= ATOL["bf16"]
