"""Pins for the oracle's 8-bit (e4m3) cache: the format's definition, a library
conversion, brute-force nearest-code search, and the quantisation error bound.

"KV cache memory systems", "Quantized cache changes attention inputs": the
cache stores 8-bit values plus separate K and V scale metadata per head; the
oracle reads that as e4m3 codes with one K and one V scale per (physical
page, kv head), stored value = code * scale.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import SMALL, page_scales

FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def _torch_encode(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def test_decode_matches_library_for_every_code():
    c = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(c)
    lib = torch.from_numpy(c).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    assert np.isnan(ours).sum() == 2  # S.1111.111 only
    assert np.array_equal(ours[~np.isnan(ours)], lib[~np.isnan(lib)])


def test_closed_forms():
    cases = {1.0: 0x38, 448.0: 0x7E, -448.0: 0xFE, 2.0 ** -9: 0x01, 2.0 ** -6: 0x08,
             0.875 * 2.0 ** -6: 0x07, 0.0: 0x00, 240.0: 0x77, 256.0: 0x78}
    for x, c in cases.items():
        assert oracle.e4m3_encode([x])[0] == c, x
    assert oracle.e4m3_encode([-0.0])[0] == 0x80
    # ties go to the even code: 2^-10 (between 0 and 2^-9), 3 * 2^-10, 1 + 1/16, 1 + 3/16
    assert oracle.e4m3_encode([2.0 ** -10, 3 * 2.0 ** -10, 1.0625, 1.1875]).tolist() == \
        [0x00, 0x02, 0x38, 0x3A]
    # saturation at the largest finite value, both signs
    big = [449.0, 464.0, 480.0, 1e6, 3e38, float("inf")]
    assert (oracle.e4m3_encode(big) == 0x7E).all()
    assert (oracle.e4m3_encode([-v for v in big]) == 0xFE).all()
    assert oracle.e4m3_encode([float("nan")])[0] & 0x7F == 0x7F


def test_round_trip_every_finite_code():
    vals = oracle.e4m3_decode(FINITE)
    assert np.array_equal(oracle.e4m3_encode(vals.astype(np.float32)), FINITE)
    # midpoints between neighbouring codes of one sign land on the even code
    for lo in range(0, 0x7E):
        for s in (0, 0x80):
            a, b = oracle.e4m3_decode(np.array([lo | s, (lo + 1) | s], np.uint8))
            mid = np.float32((a + b) / 2)
            assert float(mid) == (a + b) / 2  # exact in float32
            want = (lo if lo % 2 == 0 else lo + 1) | s
            assert oracle.e4m3_encode([mid])[0] == want, (lo, s)


def test_encode_is_the_nearest_code_brute_force():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(4000) * sc for sc in (0.01, 1.0, 30.0, 150.0)] +
                       [rng.uniform(-2.0 ** -6, 2.0 ** -6, 2000)]).astype(np.float32)
    x = np.clip(x, -448, 448)
    codes = oracle.e4m3_encode(x)
    table = oracle.e4m3_decode(FINITE)
    dist = np.abs(x.astype(np.float64)[:, None] - table[None, :])
    best = dist.min(axis=1)
    got = np.abs(x.astype(np.float64) - oracle.e4m3_decode(codes))
    assert np.array_equal(got, best)
    # and where the nearest value is unique, the code is the library's
    unique = (dist == best[:, None]).sum(axis=1) == 1
    nz = x != 0  # the library may drop the sign of values that round to zero
    assert np.array_equal(codes[unique & nz], _torch_encode(x[unique & nz]))


def test_encode_matches_library_in_range():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(50000) * rng.choice([1e-3, 0.1, 1.0, 20.0, 100.0], 50000)).astype(
        np.float32)
    x = x[np.abs(x) < 448]
    ours = oracle.e4m3_encode(x)
    lib = _torch_encode(x)
    zero = (ours & 0x7F) == 0
    assert np.array_equal(ours[~zero], lib[~zero])
    assert np.array_equal(lib[zero] & 0x7F, np.zeros(zero.sum(), np.uint8))


def _append_all(wl, scales):
    kp = np.full(wl.pool_shape(), 0xFF, dtype=np.uint8)
    vp = np.full(wl.pool_shape(), 0xFF, dtype=np.uint8)
    kb, vb = wl.empty_pool(), wl.empty_pool()
    for st in ([wl.fill] if wl.fill is not None else []) + list(wl.steps):
        sk = oracle.kv_append_e4m3(st.k_new, st.v_new, kp, vp, scales, st.block_table,
                                   st.seq_lens, st.query_start_loc, wl.block_size)
        sb = oracle.kv_append(st.k_new, st.v_new, kb, vb, st.block_table, st.seq_lens,
                              st.query_start_loc, wl.block_size)
        assert sk == 0 and sb == 0
    return kp, vp, kb, vb


@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_append_quantises_what_the_bf16_append_places(idx):
    """Placement agrees with the (pinned) bf16 append slot for slot; each code is
    the library's conversion of value / scale, saturated; unwritten slots keep
    the sentinel in both pools."""
    wl = SMALL[idx]()
    assert wl.dtype == "bf16"  # the 8-bit cache takes bf16 inputs
    scales = page_scales(wl)
    kp, vp, kb, vb = _append_all(wl, scales)
    for pool8, pool16, which in ((kp, kb, 0), (vp, vb, 1)):
        bits = pool16.view(np.uint16)
        written = bits != 0xFFFF
        assert (pool8[~written] == 0xFF).all()
        vals = oracle.widen(pool16, "bf16").astype(np.float32)
        sc = scales[:, :, which][:, :, None, None].astype(np.float32)
        y = (vals / sc).astype(np.float32)
        want = _torch_encode(np.clip(y, -448, 448))
        got = pool8[written]
        ok = want[written]
        zero = (got & 0x7F) == 0
        assert np.array_equal(got[~zero], ok[~zero])
        assert np.array_equal(ok[zero] & 0x7F, np.zeros(zero.sum(), np.uint8))


def test_gather_error_bound_and_layout():
    wl = SMALL[1]()
    scales = page_scales(wl)
    kp, vp, _, _ = _append_all(wl, scales)
    st = wl.steps[-1]
    for r in range(st.num_reqs):
        n = int(st.seq_lens[r])
        Kt, Vt = wl.request_kv(r)
        for pool, ref, which in ((kp, Kt, 0), (vp, Vt, 1)):
            got = oracle.e4m3_gather(pool, scales, which, st.block_table[r], n)
            # layout: index the pool directly through the block table
            pos = np.arange(n)
            pages = st.block_table[r][pos // wl.block_size]
            direct = oracle.e4m3_decode(pool[pages, :, pos % wl.block_size, :]) * \
                scales[pages, :, which][:, :, None].astype(np.float64)
            assert np.array_equal(got, direct)
            # value: within half a code step of value / scale, unless saturated
            x = oracle.widen(ref[:n], "bf16")
            s = np.broadcast_to(scales[pages, :, which][:, :, None].astype(np.float64), x.shape)
            y = np.abs(x / s)
            e = np.floor(np.log2(np.maximum(y, 1e-300)))
            step = np.where(y < 2.0 ** -6, 2.0 ** -9, 2.0 ** (e - 3))
            sat = y > 448
            err = np.abs(got - x) / s
            assert (err[~sat] <= step[~sat] / 2 * (1 + 1e-6) + 1e-12).all()
            assert np.array_equal(np.abs(got[sat]) / s[sat], np.full(sat.sum(), 448.0))


def test_attention_over_one_dequantised_key_is_that_value():
    wl = SMALL[1]()
    scales = page_scales(wl)
    kp, vp, _, _ = _append_all(wl, scales)
    st = wl.steps[-1]
    V = oracle.e4m3_gather(vp, scales, 1, st.block_table[0], 1)
    K = oracle.e4m3_gather(kp, scales, 0, st.block_table[0], 1)
    q = np.random.default_rng(3).standard_normal((1, wl.num_q_heads, wl.head_dim))
    out, stat = oracle.cross_attn(q, [K], [V], [1], [0, 1], wl.scale)
    assert stat == 0
    G = wl.num_q_heads // wl.num_kv_heads
    for h in range(wl.num_q_heads):
        assert np.array_equal(out[0, h], V[0, h // G])


def test_append_divides_in_float32():
    """x = 1.3671875 with scale 7 is exactly 0.1953125 = 1.5625 * 2^-3, the tie
    between codes 0x24 and 0x25 (even: 0x24); x times a float32 1/7 lands just
    above it (0x25). 2.734375 / 7 = 0.390625 is the tie 0x2C / 0x2D."""
    H_kv, D, bs = 1, 16, 16
    x = np.zeros((1, H_kv, D), dtype=np.float32)
    x[0, 0, :3] = [1.3671875, -1.3671875, 2.734375]
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)  # exact in bf16
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), x)
    kp = np.full((2, H_kv, bs, D), 0xFF, np.uint8)
    vp = kp.copy()
    scales = np.zeros((2, H_kv, 4), np.float32)
    scales[..., 0] = 7.0
    scales[..., 1] = 3.5
    assert oracle.kv_append_e4m3(bits, bits, kp, vp, scales, [[1]], [1], [0, 1], bs) == 0
    assert kp[1, 0, 0, :4].tolist() == [0x24, 0xA4, 0x2C, 0x00]
    # V: 1.3671875 / 3.5 = 0.390625 (tie -> 0x2C); 2.734375 / 3.5 = 0.78125 (tie -> 0x34)
    assert vp[1, 0, 0, :3].tolist() == [0x2C, 0xAC, 0x34]
    assert (kp[0] == 0xFF).all() and (kp[1, 0, 1:] == 0xFF).all()
