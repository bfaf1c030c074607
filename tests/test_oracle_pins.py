"""Pins for the CPU oracle: values and properties fixed by the pages or by mathematics.

Each test fails for a plausible slip in the oracle (dropped term, wrong sign,
off-by-one causal length, wrong GQA grouping, transposed operand, wrong scale).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import SMALL


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ selection


def test_select_vllm_worked_example(golden_dir):
    g = _load(golden_dir, "select_vllm_example.json")
    rows, cqsl, st = oracle.select_cross_rows(g["query_start_loc"], g["rows_per_req"])
    assert st == len(g["expected_rows"])
    assert rows.tolist() == g["expected_rows"]
    assert cqsl.tolist() == g["expected_cross_query_start_loc"]
    # the page's intermediate values, rebuilt from our rows with the library
    # routines its listing uses (bucketize -> bincount -> cumsum)
    qsl = torch.tensor(g["query_start_loc"])
    rid = torch.bucketize(torch.tensor(rows.tolist()), qsl[1:], right=True)
    assert rid.tolist() == g["expected_request_ids"]
    cnt = torch.bincount(rid, minlength=g["num_reqs"])
    assert cnt.tolist() == g["expected_counts"]


def test_select_r1r2_schedule(golden_dir):
    g = _load(golden_dir, "select_r1r2_schedule.json")
    for step in g["steps"]:
        rows, cqsl, st = oracle.select_cross_rows(step["query_start_loc"])
        assert rows.tolist() == step["expected_rows"]
        assert cqsl.tolist() == step["expected_cross_query_start_loc"]
        assert st == len(step["query_start_loc"]) - 1  # one cross row per scheduled request


def _select_via_library(qsl, rpr, rows, R):
    """cqsl rebuilt from a row list the way the page's listing does it."""
    t_rows = torch.tensor(rows.tolist(), dtype=torch.int64)
    t_qsl = torch.tensor(qsl.tolist(), dtype=torch.int64)
    rid = torch.bucketize(t_rows, t_qsl[1:], right=True)
    cnt = torch.bincount(rid, minlength=R)
    return np.concatenate([[0], torch.cumsum(cnt, 0).numpy()]).astype(np.int32), cnt.numpy()


@pytest.mark.parametrize("seed", range(20))
def test_select_random_matches_library_rebuild(seed):
    rng = np.random.default_rng(seed)
    R = int(rng.integers(0, 40))
    qlen = rng.integers(0, 9, size=R)
    qlen[rng.random(R) < 0.5] = 1  # many decodes
    qsl = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    rpr = None if seed % 2 == 0 else rng.integers(0, 5, size=R).astype(np.int32)
    rows, cqsl, st = oracle.select_cross_rows(qsl, rpr)
    want = np.ones(R, np.int64) if rpr is None else rpr.astype(np.int64)
    k = np.minimum(want, qlen)
    assert st == int(k.sum())
    lib_cqsl, cnt = _select_via_library(qsl, rpr, rows, R)
    assert cqsl.tolist() == lib_cqsl.tolist()
    assert cnt.tolist() == k.tolist()
    for r in range(R):
        mine = rows[cqsl[r]:cqsl[r + 1]].tolist()
        # the trailing k_r scheduled tokens of request r, in order
        assert mine == list(range(qsl[r + 1] - k[r], qsl[r + 1]))


def test_select_edge_cases():
    rows, cqsl, st = oracle.select_cross_rows([0])  # no requests
    assert rows.tolist() == [] and cqsl.tolist() == [0] and st == 0
    rows, cqsl, st = oracle.select_cross_rows([0, 0, 3, 3])  # q_len 0 requests give no row
    assert rows.tolist() == [2] and cqsl.tolist() == [0, 0, 1, 1]
    rows, cqsl, st = oracle.select_cross_rows([0, 2, 5], [7, 0])  # clamp to q_len; zero rows
    assert rows.tolist() == [0, 1] and cqsl.tolist() == [0, 2, 2]
    _, _, st = oracle.select_cross_rows([0, 3, 2])  # decreasing offsets are an error
    assert st == -1
    _, _, st = oracle.select_cross_rows([0, 3], [-1])
    assert st == -1


# --------------------------------------------------------------------- append


def test_append_hand_worked(golden_dir):
    g = _load(golden_dir, "append_tiny.json")
    bs, nb = g["block_size"], g["num_blocks"]
    T = g["query_start_loc"][-1]
    k_new = (100.0 + np.arange(T, dtype=np.float32)).reshape(T, 1, 1)
    v_new = k_new + 100.0
    kp = np.full((nb, 1, bs, 1), -1.0, np.float32)
    vp = np.full((nb, 1, bs, 1), -1.0, np.float32)
    skipped = oracle.kv_append(k_new, v_new, kp, vp, g["block_table"], g["seq_lens"],
                               g["query_start_loc"], bs)
    assert skipped == 0
    exp = np.array(g["expected_k_pool"], np.float32)
    assert np.array_equal(kp[:, 0, :, 0], exp)
    assert np.array_equal(vp[:, 0, :, 0], np.where(exp >= 0, exp + 100, -1))


def test_append_out_of_range_is_skipped():
    kp = np.full((2, 1, 4, 1), -1.0, np.float32)
    vp = kp.copy()
    k_new = np.arange(3, dtype=np.float32).reshape(3, 1, 1)
    # request 0: page id 7 does not exist; request 1: position 4 needs a 2nd block it lacks
    skipped = oracle.kv_append(k_new, k_new, kp, vp, [[7], [1]], [1, 5], [0, 1, 3], 4)
    assert skipped == 2
    assert kp[1, 0, 3, 0] == 1.0 and (kp[0] == -1).all()


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_append_readback_brute_force(idx):
    """Fill + step appended by the oracle, read back slot by slot through the block table."""
    wl = SMALL[idx]()
    kp, vp = wl.empty_pool(), wl.empty_pool()
    written = np.zeros(kp.shape[:3], dtype=np.int64)
    steps = ([wl.fill] if wl.fill is not None else []) + wl.steps
    for st in steps:
        assert oracle.kv_append(st.k_new, st.v_new, kp, vp, st.block_table, st.seq_lens,
                                st.query_start_loc, wl.block_size) == 0
    bs = wl.block_size
    final = wl.steps[-1]
    for b, r in enumerate(final.req_ids):
        K, V = wl.request_kv(r)
        for pos in range(int(final.seq_lens[b])):
            page = final.block_table[b, pos // bs]
            assert np.array_equal(kp[page, :, pos % bs, :], K[pos])
            assert np.array_equal(vp[page, :, pos % bs, :], V[pos])
            written[page, :, pos % bs] = 1
    # every slot not holding a token still holds the sentinel bytes
    untouched = kp.view(np.uint8).reshape(kp.shape[:3] + (-1,))[written == 0]
    assert (untouched == 0xFF).all()


def test_append_page_permutation_only_moves_pages():
    a = SMALL[1]()
    b = SMALL[1]()
    # re-permute b's physical pages: the same logical contents must read back
    rng = np.random.default_rng(7)
    perm = rng.permutation(b.num_blocks).astype(np.int32)
    for st in [b.fill] + b.steps:
        st.block_table = perm[st.block_table]
    pools = []
    for wl in (a, b):
        kp, vp = wl.empty_pool(), wl.empty_pool()
        for st in [wl.fill] + wl.steps:
            oracle.kv_append(st.k_new, st.v_new, kp, vp, st.block_table, st.seq_lens,
                             st.query_start_loc, wl.block_size)
        pools.append(kp)
    assert np.array_equal(pools[1][perm], pools[0])


# ------------------------------------------------------------------ attention


def _one_request(K, V, q, seq_len=None, scale=None):
    """q [rows, H_q, D] for one request whose trailing rows are queried."""
    n = K.shape[0] if seq_len is None else seq_len
    rows = q.shape[0]
    scale = 1.0 / math.sqrt(q.shape[-1]) if scale is None else scale
    out, st = oracle.cross_attn(q, [K], [V], [n], [0, rows], scale)
    assert st == 0
    return out


def test_attn_single_key_returns_v_exactly():
    rng = np.random.default_rng(0)
    K = rng.standard_normal((1, 2, 64))
    V = rng.standard_normal((1, 2, 64))
    q = rng.standard_normal((1, 8, 64)) * 10
    out = _one_request(K, V, q)
    for h in range(8):
        assert np.array_equal(out[0, h], V[0, h // 4])


def test_attn_equal_scores_give_mean():
    rng = np.random.default_rng(1)
    K = rng.standard_normal((37, 1, 32))
    V = rng.standard_normal((37, 1, 32))
    q = np.zeros((1, 3, 32))
    out = _one_request(K, V, q)
    np.testing.assert_allclose(out[0], np.broadcast_to(V[:, 0].mean(0), (3, 32)), atol=1e-15, rtol=0)


def test_attn_two_keys_closed_form():
    # s1 - s2 = scale * q.(k1 - k2); weight of key 1 is the logistic function of it
    q = np.array([[[1.0, 0.0]]])
    K = np.array([[[1.0, 0.0]], [[0.0, 1.0]]])
    V = np.array([[[1.0, 2.0]], [[3.0, 4.0]]])
    sig = 0.66976155  # logistic(1/sqrt(2)), worked by hand
    out = _one_request(K, V, q, scale=1 / math.sqrt(2))
    np.testing.assert_allclose(out[0, 0], [sig * 1 + (1 - sig) * 3, sig * 2 + (1 - sig) * 4],
                               atol=1e-8)
    # doubling the scale doubles the logit gap: logistic(sqrt 2) = 0.80443
    out2 = _one_request(K, V, q, scale=math.sqrt(2))
    sig2 = 0.80442968
    np.testing.assert_allclose(out2[0, 0], [sig2 + (1 - sig2) * 3, 2 * sig2 + (1 - sig2) * 4],
                               atol=1e-7)


def test_attn_dominant_key_saturates():
    rng = np.random.default_rng(2)
    K = rng.standard_normal((10, 1, 16)) * 0.01
    q = np.zeros((1, 1, 16))
    q[0, 0, 0] = 1.0
    K[6, 0, 0] = 5000.0  # score 5000/4 above all others
    V = rng.standard_normal((10, 1, 16))
    out = _one_request(K, V, q)
    np.testing.assert_allclose(out[0, 0], V[6, 0], atol=1e-300, rtol=1e-15)


def test_attn_gqa_grouping_is_contiguous():
    H_q, H_kv, D = 8, 2, 16
    rng = np.random.default_rng(3)
    K = rng.standard_normal((20, H_kv, D))
    V = np.zeros((20, H_kv, D))
    V[:, 1, :] = 1.0  # kv head 1 carries ones, kv head 0 zeros
    q = rng.standard_normal((1, H_q, D))
    out = _one_request(K, V, q)
    for h in range(H_q):
        assert np.allclose(out[0, h], 0.0 if h < 4 else 1.0, atol=1e-15)


def test_attn_causal_prefix_invariance():
    """Keys after the query position never change its output (exact in f64)."""
    rng = np.random.default_rng(4)
    K = rng.standard_normal((50, 2, 32))
    V = rng.standard_normal((50, 2, 32))
    q = rng.standard_normal((1, 4, 32))
    base = _one_request(K[:30], V[:30], q, seq_len=30)
    K2, V2 = K.copy(), V.copy()
    K2[30:] = 1e3
    V2[30:] = -7.0
    again = _one_request(K2, V2, q, seq_len=30)
    assert np.array_equal(base, again)
    longer = _one_request(K2, V2, q, seq_len=31)
    assert not np.allclose(base, longer)


def _sdpa_f64(q_rows, K, V, kv_lens, scale):
    """Library special case: torch SDPA (float64, CPU) with an explicit mask per row."""
    qt = torch.from_numpy(q_rows).permute(1, 0, 2)[None]  # [1, H_q, rows, D]
    kt = torch.from_numpy(K).permute(1, 0, 2)[None]
    vt = torch.from_numpy(V).permute(1, 0, 2)[None]
    n = K.shape[0]
    mask = torch.zeros(q_rows.shape[0], n, dtype=torch.bool)
    for i, L in enumerate(kv_lens):
        mask[i, :L] = True
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale,
                                                         enable_gqa=True)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("H_q,H_kv", [(4, 1), (8, 2), (16, 1), (6, 3)])
def test_attn_matches_library_sdpa(H_q, H_kv):
    rng = np.random.default_rng(H_q * 10 + H_kv)
    seq, rows, D = 45, 5, 32
    K = rng.standard_normal((seq, H_kv, D))
    V = rng.standard_normal((seq, H_kv, D))
    q = rng.standard_normal((rows, H_q, D))
    out = _one_request(K, V, q, seq_len=seq)
    # bottom-right causal: trailing row i of `rows` sees seq - rows + i + 1 keys
    ref = _sdpa_f64(q, K, V, [seq - rows + i + 1 for i in range(rows)], 1 / math.sqrt(D))
    np.testing.assert_allclose(out, ref, atol=1e-12, rtol=0)


def test_attn_pure_prefill_matches_library_causal():
    """A request whose whole prompt is scheduled: every row = torch's is_causal attention."""
    rng = np.random.default_rng(5)
    n, H, D = 24, 4, 16
    K = rng.standard_normal((n, 2, D))
    V = rng.standard_normal((n, 2, D))
    q = rng.standard_normal((n, H, D))
    out = _one_request(K, V, q, seq_len=n)
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(K).permute(1, 0, 2)[None]
    vt = torch.from_numpy(V).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True,
                                                           enable_gqa=True)[0].permute(1, 0, 2)
    np.testing.assert_allclose(out, ref.numpy(), atol=1e-12, rtol=0)


def test_attn_prefill_skip_invariance():
    """Computing every scheduled row and keeping the last one per request equals
    computing only the selected rows (the cross-decoder 'vertical line')."""
    wl = SMALL[2]()
    st = wl.steps[0]
    qsl = st.query_start_loc
    q_len = np.diff(qsl)
    rows_all, cqsl_all, _ = oracle.select_cross_rows(qsl, q_len)  # every scheduled token
    rows_sel, cqsl_sel, _ = oracle.select_cross_rows(qsl)  # one per request
    assert rows_all.tolist() == list(range(st.num_tokens))
    rng = np.random.default_rng(6)
    q_all = rng.standard_normal((st.num_tokens, wl.num_q_heads, wl.head_dim))
    Ks, Vs = [], []
    for r in st.req_ids:
        K, V = wl.request_kv(r)
        Ks.append(oracle.widen(K, wl.dtype))
        Vs.append(oracle.widen(V, wl.dtype))
    out_all, s1 = oracle.cross_attn(q_all, Ks, Vs, st.seq_lens, cqsl_all, wl.scale)
    out_sel, s2 = oracle.cross_attn(q_all[rows_sel], Ks, Vs, st.seq_lens, cqsl_sel, wl.scale)
    assert s1 == 0 and s2 == 0
    assert np.array_equal(out_all[rows_sel], out_sel)


def test_attn_bad_rows_are_reported():
    K = np.ones((4, 1, 8))
    q = np.ones((1, 1, 8))
    out, st = oracle.cross_attn(q, [K], [K], [0], [0, 1], 1.0)  # seq_len 0: no key to attend
    assert st == -1 and (out == 0).all()
    out, st = oracle.cross_attn(q, [K], [K], [9], [0, 1], 1.0)  # more keys than stored
    assert st == -1


def test_widen_bf16_exact():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0001, 0x7F7F], dtype=np.uint16)
    got = oracle.widen(bits, "bf16")
    assert got[0] == 1.0 and got[1] == -1.0
    assert got[2] == 3.140625
    assert got[3] == 2.0 ** -133  # smallest bf16 subnormal
    assert got[4] == (2 - 2 ** -7) * 2.0 ** 127  # largest finite bf16


def test_attn_row_wrapper_closed_forms():
    """The single-row entry point, directly: only the first kv_len keys count
    (two-key logistic weight), and one key returns V exactly per kv head."""
    q = np.array([[1.0, 0.0]])
    K = np.array([[[1.0, 0.0]], [[0.0, 1.0]], [[50.0, 0.0]]])  # the third key lies past kv_len
    V = np.array([[[1.0, 2.0]], [[3.0, 4.0]], [[-9.0, -9.0]]])
    sig = 0.66976155  # logistic(1/sqrt(2)), worked by hand
    out = oracle.attn_row(q, K, V, 2, 1 / math.sqrt(2))
    np.testing.assert_allclose(out[0], [sig * 1 + (1 - sig) * 3, sig * 2 + (1 - sig) * 4], atol=1e-8)
    rng = np.random.default_rng(4)
    K1 = rng.standard_normal((3, 2, 8))
    V1 = rng.standard_normal((3, 2, 8))
    q1 = rng.standard_normal((6, 8)) * 10
    out1 = oracle.attn_row(q1, K1, V1, 1, 0.3)
    for h in range(6):
        assert np.array_equal(out1[h], V1[0, h // 3])
