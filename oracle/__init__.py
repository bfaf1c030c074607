"""CPU oracle for the YOCO cross-decoder hot path — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never does, and this
package never imports the CUDA library: the two share no code.

The arithmetic lives in ``yoco_oracle.c`` (float64, explicit loops); this
module only marshals numpy arrays into it and widens stored bf16/f32 values
to float64 exactly.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

import numpy as np

from . import build as _build

_lib = None

_i32p = ctypes.POINTER(ctypes.c_int32)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_f64p = ctypes.POINTER(ctypes.c_double)


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.oracle_select_cross_rows.restype = ctypes.c_int64
        L.oracle_select_cross_rows.argtypes = [_i32p, _i32p, ctypes.c_int32, _i32p, _i32p]
        L.oracle_kv_append.restype = ctypes.c_int64
        L.oracle_kv_append.argtypes = [_u8p, _u8p, _u8p, _u8p, _i32p, ctypes.c_int32, _i32p, _i32p,
                                       ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]
        L.oracle_attn_row.restype = None
        L.oracle_attn_row.argtypes = [_f64p, _f64p, _f64p, ctypes.c_int64, ctypes.c_int32,
                                      ctypes.c_int32, ctypes.c_int32, ctypes.c_double, _f64p, _f64p]
        L.oracle_cross_attn.restype = ctypes.c_int32
        L.oracle_cross_attn.argtypes = [_f64p, ctypes.POINTER(_f64p), ctypes.POINTER(_f64p), _i32p,
                                        _i32p, ctypes.c_int32, _i32p, ctypes.c_int64,
                                        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_double, _f64p, ctypes.POINTER(ctypes.c_int64),
                                        ctypes.c_int32]
        L.oracle_e4m3_encode_array.restype = None
        L.oracle_e4m3_encode_array.argtypes = [ctypes.c_void_p, ctypes.c_int64, _u8p]
        L.oracle_e4m3_decode_array.restype = None
        L.oracle_e4m3_decode_array.argtypes = [_u8p, ctypes.c_int64, _f64p]
        L.oracle_kv_append_e4m3.restype = ctypes.c_int64
        L.oracle_kv_append_e4m3.argtypes = [ctypes.c_void_p, ctypes.c_void_p, _u8p, _u8p,
                                            ctypes.c_void_p, _i32p, ctypes.c_int32, _i32p, _i32p,
                                            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                            ctypes.c_int32, ctypes.c_int32]
        L.oracle_e4m3_gather.restype = ctypes.c_int32
        L.oracle_e4m3_gather.argtypes = [_u8p, ctypes.c_void_p, ctypes.c_int32, _i32p,
                                         ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_int32, ctypes.c_int32, _f64p]
        _lib = L
    return _lib


def _p(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def widen(x: np.ndarray, dtype: str) -> np.ndarray:
    """Stored values -> float64, exactly (bf16 bits are the top half of an f32)."""
    if dtype == "bf16":
        bits = np.ascontiguousarray(x).view(np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    raise ValueError(dtype)


def select_cross_rows(query_start_loc, rows_per_req=None) -> Tuple[np.ndarray, np.ndarray, int]:
    """Cross-decoder row list and cross query_start_loc; returns (rows, cqsl, status).

    status is the row count, or -1 for a negative q_len / rows_per_req.
    """
    qsl = _i32(query_start_loc)
    R = qsl.shape[0] - 1
    cap = max(int(qsl[-1] - qsl[0]) if R > 0 else 0, 0)
    rpr = None if rows_per_req is None else _i32(rows_per_req)
    if rpr is not None:
        cap = max(cap, int(np.clip(rpr, 0, None).sum()))
    rows = np.zeros(max(cap, 1), dtype=np.int32)
    cqsl = np.zeros(R + 1, dtype=np.int32)
    n = lib().oracle_select_cross_rows(_p(qsl, _i32p), None if rpr is None else _p(rpr, _i32p),
                                       R, _p(rows, _i32p), _p(cqsl, _i32p))
    count = int(cqsl[-1]) if R >= 0 else 0
    return rows[:count].copy(), cqsl, int(n)


def kv_append(k_new: np.ndarray, v_new: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray,
              block_table, seq_lens, query_start_loc, block_size: int) -> int:
    """In-place append into numpy pools ``[num_blocks, H_kv, bs, D]``; returns skipped count."""
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    num_blocks, H_kv, bs, D = k_pool.shape
    assert bs == block_size
    esz = k_pool.dtype.itemsize
    kn = np.ascontiguousarray(k_new).view(np.uint8)
    vn = np.ascontiguousarray(v_new).view(np.uint8)
    bt = _i32(block_table)
    if bt.ndim == 1:
        bt = bt.reshape(1, -1)
    qsl, sl = _i32(query_start_loc), _i32(seq_lens)
    R = qsl.shape[0] - 1
    max_blocks = bt.shape[1] if bt.size else 1
    return int(lib().oracle_kv_append(_p(kn, _u8p), _p(vn, _u8p), _p(k_pool.view(np.uint8), _u8p),
                                      _p(v_pool.view(np.uint8), _u8p), _p(bt, _i32p), max_blocks,
                                      _p(sl, _i32p), _p(qsl, _i32p), R, num_blocks, bs, H_kv, D, esz))


def attn_row(q: np.ndarray, K: np.ndarray, V: np.ndarray, kv_len: int, scale: float) -> np.ndarray:
    """One row: q [H_q, D], K/V [>=kv_len, H_kv, D] (float64) -> out [H_q, D]."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    H_q, D = q.shape
    H_kv = K.shape[1]
    assert K.shape[0] >= kv_len and V.shape[0] >= kv_len
    out = np.zeros((H_q, D), dtype=np.float64)
    w = np.zeros(max(kv_len, 1), dtype=np.float64)
    lib().oracle_attn_row(_p(q, _f64p), _p(K, _f64p), _p(V, _f64p), kv_len, H_q, H_kv, D,
                          float(scale), _p(out, _f64p), _p(w, _f64p))
    return out


def cross_attn(q: np.ndarray, K_req: Sequence[np.ndarray], V_req: Sequence[np.ndarray], seq_lens,
               cross_query_start_loc, scale: float, rows: Optional[Sequence[int]] = None,
               nthreads: int = 1) -> Tuple[np.ndarray, int]:
    """Attention for the selected rows (all rows if ``rows`` is None).

    q: [num_rows, H_q, D] float64; K_req[r]/V_req[r]: [len_r, H_kv, D] float64.
    Returns (out [len(rows), H_q, D], status 0 or -1).
    """
    q = np.ascontiguousarray(q, dtype=np.float64)
    cq = _i32(cross_query_start_loc)
    sl = _i32(seq_lens)
    R = cq.shape[0] - 1
    num_rows, H_q, D = q.shape
    row_list = _i32(np.arange(num_rows) if rows is None else rows)
    Ks = [np.ascontiguousarray(k, dtype=np.float64) for k in K_req]
    Vs = [np.ascontiguousarray(v, dtype=np.float64) for v in V_req]
    assert len(Ks) >= R and len(Vs) >= R
    H_kv = Ks[0].shape[1] if Ks else 1
    cap = np.array([min(Ks[r].shape[0], Vs[r].shape[0]) for r in range(R)] or [0], dtype=np.int64)
    kp = (_f64p * max(R, 1))(*[_p(k, _f64p) for k in Ks[:R]])
    vp = (_f64p * max(R, 1))(*[_p(v, _f64p) for v in Vs[:R]])
    out = np.zeros((row_list.shape[0], H_q, D), dtype=np.float64)
    st = lib().oracle_cross_attn(_p(q, _f64p), kp, vp, _p(sl, _i32p), _p(cq, _i32p), R,
                                 _p(row_list, _i32p), row_list.shape[0], H_q, H_kv, D, float(scale),
                                 _p(out, _f64p), cap.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                 max(1, int(nthreads)))
    return out, int(st)


# ------------------------------------------------------------------ e4m3 cache

def e4m3_encode(x) -> np.ndarray:
    """float32 values -> e4m3 codes (nearest, ties to even, saturating at +-448)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.zeros(x.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode_array(x.ctypes.data, x.size, _p(out, _u8p))
    return out


def e4m3_decode(codes) -> np.ndarray:
    """e4m3 codes -> float64 values (NaN for the two NaN codes)."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.zeros(c.shape, dtype=np.float64)
    lib().oracle_e4m3_decode_array(_p(c, _u8p), c.size, _p(out, _f64p))
    return out


def kv_append_e4m3(k_new: np.ndarray, v_new: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray,
                   scales: np.ndarray, block_table, seq_lens, query_start_loc,
                   block_size: int) -> int:
    """Quantising append: bf16 bits [T, H_kv, D] into uint8 pools [num_blocks, H_kv, bs, D];
    scales float32 [num_blocks, H_kv, 4] = (k_scale, v_scale, -, -). Returns skipped count."""
    assert k_pool.dtype == np.uint8 and v_pool.dtype == np.uint8
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    num_blocks, H_kv, bs, D = k_pool.shape
    assert bs == block_size
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    assert sc.shape == (num_blocks, H_kv, 4)
    kn = np.ascontiguousarray(k_new).view(np.uint16)
    vn = np.ascontiguousarray(v_new).view(np.uint16)
    bt = _i32(block_table)
    if bt.ndim == 1:
        bt = bt.reshape(1, -1)
    qsl, sl = _i32(query_start_loc), _i32(seq_lens)
    R = qsl.shape[0] - 1
    max_blocks = bt.shape[1] if bt.size else 1
    return int(lib().oracle_kv_append_e4m3(kn.ctypes.data, vn.ctypes.data, _p(k_pool, _u8p),
                                           _p(v_pool, _u8p), sc.ctypes.data, _p(bt, _i32p),
                                           max_blocks, _p(sl, _i32p), _p(qsl, _i32p), R,
                                           num_blocks, bs, H_kv, D))


def e4m3_gather(pool: np.ndarray, scales: np.ndarray, which: int, bt_row,
                n_tokens: int) -> np.ndarray:
    """Dequantised [n_tokens, H_kv, D] float64 of one request (which: 0 = K scale, 1 = V)."""
    num_blocks, H_kv, bs, D = pool.shape
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    bt = _i32(bt_row)
    out = np.zeros((max(n_tokens, 0), H_kv, D), dtype=np.float64)
    st = lib().oracle_e4m3_gather(_p(np.ascontiguousarray(pool), _u8p), sc.ctypes.data, which,
                                  _p(bt, _i32p), n_tokens, num_blocks, bs, H_kv, D,
                                  _p(out, _f64p))
    if st != 0:
        raise ValueError("page index out of range")
    return out
