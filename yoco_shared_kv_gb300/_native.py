"""ctypes binding of ``include/yoco_kv.h`` — argument marshalling only.

Every function here has the name of the C entry point it wraps, takes torch
tensors that already live on the GPU, checks their dtype/shape/contiguity,
and passes raw pointers and sizes through. All arithmetic happens in the
CUDA library. There is no fallback: if the library is not built, importing
this module raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libyoco_kv.so")

YOCO_OK, YOCO_ERR_INVALID_ARG, YOCO_ERR_UNSUPPORTED, YOCO_ERR_WORKSPACE, YOCO_ERR_CUDA = range(5)
YOCO_F32, YOCO_BF16, YOCO_E4M3 = 0, 1, 2
YOCO_ATTN_REVERSE = 0x1
YOCO_ATTN_OVERLAP = 0x2
YOCO_ATTN_KEEP_TAIL = 0x4
YOCO_ATTN_PLANNED = 0x8
DEVERR_PAGE_RANGE = 0x1
DEVERR_POS_RANGE = 0x2
DEVERR_EMPTY_ROW = 0x4
DEVERR_OFFSETS = 0x8
DEVERR_TIMEOUT = 0x10
DEVERR_SCALE = 0x20
DEVERR_PLAN = 0x40

EXPORTED = ("yoco_kv_append", "yoco_select_cross_rows", "yoco_cross_attn_workspace_size",
            "yoco_cross_attn_paged", "yoco_set_l2_window", "yoco_status_string", "yoco_version",
            "yoco_last_cuda_error", "yoco_last_cuda_error_string",
            "yoco_cross_attn_paged_noalloc", "yoco_cross_attn_noalloc_capacity",
            "yoco_selftest_wait_timeout", "yoco_cross_decoder_bytes", "yoco_kv_append_e4m3",
            "yoco_cross_attn_paged_e4m3", "yoco_cross_decode_step", "yoco_cross_attn_plan")


class YocoError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = f"{fn} failed: {status_name(status)} (status {status})"
        if status == YOCO_ERR_CUDA:
            msg += f": {lib.yoco_last_cuda_error_string().decode()}"
        super().__init__(msg)
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"CUDA library not built: {LIB_PATH} is missing "
                          "(run yoco_shared_kv_gb300.build.build())")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    L.yoco_kv_append.restype = ctypes.c_int
    L.yoco_kv_append.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32,
                                 ctypes.c_int, vp, vp]
    L.yoco_select_cross_rows.restype = ctypes.c_int
    L.yoco_select_cross_rows.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp]
    L.yoco_cross_attn_workspace_size.restype = sz
    L.yoco_cross_attn_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.c_int]
    L.yoco_cross_attn_paged.restype = ctypes.c_int
    L.yoco_cross_attn_paged.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32,
                                        i32, i32, i32, ctypes.c_float, ctypes.c_int,
                                        ctypes.c_uint32, vp, sz, vp, vp]
    L.yoco_set_l2_window.restype = ctypes.c_int
    L.yoco_set_l2_window.argtypes = [vp, vp, sz, ctypes.c_float]
    L.yoco_status_string.restype = ctypes.c_char_p
    L.yoco_status_string.argtypes = [ctypes.c_int]
    L.yoco_version.restype = ctypes.c_int32
    L.yoco_version.argtypes = []
    L.yoco_last_cuda_error.restype = ctypes.c_int32
    L.yoco_last_cuda_error.argtypes = []
    L.yoco_last_cuda_error_string.restype = ctypes.c_char_p
    L.yoco_last_cuda_error_string.argtypes = []
    L.yoco_cross_attn_paged_noalloc.restype = ctypes.c_int
    L.yoco_cross_attn_paged_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32,
                                                i32, i32, i32, i32, i32, ctypes.c_float,
                                                ctypes.c_int, vp, vp]
    L.yoco_cross_attn_noalloc_capacity.restype = sz
    L.yoco_cross_attn_noalloc_capacity.argtypes = []
    L.yoco_selftest_wait_timeout.restype = ctypes.c_int
    L.yoco_selftest_wait_timeout.argtypes = [vp, ctypes.c_uint32, vp]
    L.yoco_cross_decoder_bytes.restype = ctypes.c_int64
    L.yoco_cross_decoder_bytes.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, ctypes.c_int,
                                           vp]
    L.yoco_kv_append_e4m3.restype = ctypes.c_int
    L.yoco_kv_append_e4m3.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32,
                                      i32, vp, vp]
    L.yoco_cross_decode_step.restype = ctypes.c_int
    L.yoco_cross_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32,
                                         i32, i32, i32, i32, i32, ctypes.c_float, ctypes.c_int,
                                         ctypes.c_uint32, vp, sz, vp, vp]
    L.yoco_cross_attn_plan.restype = ctypes.c_int
    L.yoco_cross_attn_plan.argtypes = [vp, i32, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32,
                                       ctypes.c_int, ctypes.c_uint32, vp, sz, vp, vp]
    L.yoco_cross_attn_paged_e4m3.restype = ctypes.c_int
    L.yoco_cross_attn_paged_e4m3.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32,
                                             i32, i32, i32, i32, i32, ctypes.c_float,
                                             ctypes.c_uint32, vp, sz, vp, vp]
    return L


lib = _load()


def status_name(status: int) -> str:
    return lib.yoco_status_string(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != YOCO_OK:
        raise YocoError(fn, status)


def dtype_code(t: torch.dtype) -> int:
    """bf16 / fp32 caches; torch.float8_e4m3fn (or uint8) names the e4m3 cache."""
    if t == torch.bfloat16:
        return YOCO_BF16
    if t == torch.float32:
        return YOCO_F32
    if t in (torch.float8_e4m3fn, torch.uint8):
        return YOCO_E4M3
    raise ValueError(f"unsupported dtype {t}")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _i32(t: torch.Tensor, name: str) -> int:
    if t.dtype != torch.int32:
        raise ValueError(f"{name} must be int32")
    return _ptr(t)


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def yoco_kv_append(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                   v_cache: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                   query_start_loc: torch.Tensor, err_word: Optional[torch.Tensor] = None,
                   stream=None) -> None:
    """Append ``k_new/v_new [T, H_kv, D]`` into pools ``[num_blocks, H_kv, bs, D]``."""
    num_blocks, H_kv, bs, D = k_cache.shape
    assert v_cache.shape == k_cache.shape and k_new.shape == v_new.shape
    assert k_new.dtype == k_cache.dtype == v_cache.dtype == v_new.dtype
    T = k_new.shape[0]
    assert k_new.shape[1:] == (H_kv, D)
    R = query_start_loc.shape[0] - 1
    _check("yoco_kv_append", lib.yoco_kv_append(
        _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _i32(block_table, "block_table"),
        block_table.shape[1], _i32(seq_lens, "seq_lens"), _i32(query_start_loc, "query_start_loc"),
        R, T, num_blocks, bs, H_kv, D, dtype_code(k_cache.dtype),
        None if err_word is None else _i32(err_word, "err_word"), _stream(stream)))


def yoco_select_cross_rows(query_start_loc: torch.Tensor, rows_per_req: Optional[torch.Tensor],
                           row_indices: torch.Tensor, cross_query_start_loc: torch.Tensor,
                           num_rows: torch.Tensor, err_word: Optional[torch.Tensor] = None,
                           stream=None) -> None:
    R = query_start_loc.shape[0] - 1
    assert cross_query_start_loc.shape[0] == R + 1
    _check("yoco_select_cross_rows", lib.yoco_select_cross_rows(
        _i32(query_start_loc, "query_start_loc"),
        None if rows_per_req is None else _i32(rows_per_req, "rows_per_req"), R,
        _i32(row_indices, "row_indices"), _i32(cross_query_start_loc, "cross_query_start_loc"),
        _i32(num_rows, "num_rows"), None if err_word is None else _i32(err_word, "err_word"),
        _stream(stream)))


def yoco_cross_attn_workspace_size(max_rows: int, num_q_heads: int, num_kv_heads: int,
                                   head_dim: int, block_size: int, max_seq_len: int,
                                   dtype: torch.dtype) -> int:
    return int(lib.yoco_cross_attn_workspace_size(max_rows, num_q_heads, num_kv_heads, head_dim,
                                                  block_size, max_seq_len, dtype_code(dtype)))


def yoco_cross_attn_paged(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                          out: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                          cross_query_start_loc: torch.Tensor, max_seq_len: int, scale: float,
                          workspace: Optional[torch.Tensor], err_word: Optional[torch.Tensor] = None,
                          stream=None, max_rows: Optional[int] = None, flags: int = 0) -> None:
    """One layer: ``q/out [max_rows, H_q, D]`` against pools ``[num_blocks, H_kv, bs, D]``."""
    num_blocks, H_kv, bs, D = k_cache.shape
    rows_cap, H_q, Dq = q.shape
    assert Dq == D and out.shape == q.shape and out.dtype == q.dtype == k_cache.dtype
    R = cross_query_start_loc.shape[0] - 1
    max_rows = rows_cap if max_rows is None else max_rows
    assert max_rows <= rows_cap
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("yoco_cross_attn_paged", lib.yoco_cross_attn_paged(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _i32(block_table, "block_table"),
        block_table.shape[1], _i32(seq_lens, "seq_lens"),
        _i32(cross_query_start_loc, "cross_query_start_loc"), R, max_rows, int(max_seq_len), H_q,
        H_kv, D, bs, num_blocks, float(scale), dtype_code(q.dtype), int(flags), _ptr(workspace),
        ws_bytes, None if err_word is None else _i32(err_word, "err_word"), _stream(stream)))


def yoco_cross_attn_plan(block_table: torch.Tensor, seq_lens: torch.Tensor,
                         cross_query_start_loc: torch.Tensor, max_seq_len: int, max_rows: int,
                         num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                         num_blocks: int, dtype: torch.dtype, workspace: Optional[torch.Tensor],
                         err_word: Optional[torch.Tensor] = None, stream=None,
                         flags: int = 0) -> None:
    """The step's plan into ``workspace``; later layers pass ``YOCO_ATTN_PLANNED``."""
    R = cross_query_start_loc.shape[0] - 1
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("yoco_cross_attn_plan", lib.yoco_cross_attn_plan(
        _i32(block_table, "block_table"), block_table.shape[1], _i32(seq_lens, "seq_lens"),
        _i32(cross_query_start_loc, "cross_query_start_loc"), R, int(max_rows), int(max_seq_len),
        int(num_q_heads), int(num_kv_heads), int(head_dim), int(block_size), int(num_blocks),
        dtype_code(dtype), int(flags), _ptr(workspace), ws_bytes,
        None if err_word is None else _i32(err_word, "err_word"), _stream(stream)))


def yoco_cross_attn_paged_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                  out: torch.Tensor, block_table: torch.Tensor,
                                  seq_lens: torch.Tensor, cross_query_start_loc: torch.Tensor,
                                  max_seq_len: int, scale: float,
                                  err_word: Optional[torch.Tensor] = None, stream=None,
                                  max_rows: Optional[int] = None) -> None:
    """yoco_cross_attn_paged with the library's fixed scratch array: no workspace, no allocation."""
    num_blocks, H_kv, bs, D = k_cache.shape
    rows_cap, H_q, Dq = q.shape
    assert Dq == D and out.shape == q.shape and out.dtype == q.dtype == k_cache.dtype
    R = cross_query_start_loc.shape[0] - 1
    max_rows = rows_cap if max_rows is None else max_rows
    assert max_rows <= rows_cap
    _check("yoco_cross_attn_paged_noalloc", lib.yoco_cross_attn_paged_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _i32(block_table, "block_table"),
        block_table.shape[1], _i32(seq_lens, "seq_lens"),
        _i32(cross_query_start_loc, "cross_query_start_loc"), R, max_rows, int(max_seq_len), H_q,
        H_kv, D, bs, num_blocks, float(scale), dtype_code(q.dtype),
        None if err_word is None else _i32(err_word, "err_word"), _stream(stream)))


def yoco_cross_attn_noalloc_capacity() -> int:
    return int(lib.yoco_cross_attn_noalloc_capacity())


def yoco_cross_decoder_bytes(query_start_loc, rows_per_req, seq_lens, layers: int,
                             num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                             dtype: torch.dtype):
    """Traffic model on host arrays: (total bytes, per-request bytes)."""
    import numpy as np
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    rpr = None if rows_per_req is None else np.ascontiguousarray(rows_per_req, dtype=np.int32)
    R = qsl.shape[0] - 1
    per = np.zeros(max(R, 1), dtype=np.int64)
    tot = lib.yoco_cross_decoder_bytes(
        qsl.ctypes.data, None if rpr is None else rpr.ctypes.data, sl.ctypes.data, R, layers,
        num_q_heads, num_kv_heads, head_dim, block_size, dtype_code(dtype), per.ctypes.data)
    if tot < 0:
        raise ValueError("invalid arguments")
    return int(tot), per[:R]


def yoco_selftest_wait_timeout(err_word: torch.Tensor, limit_us: int = 20000, stream=None) -> None:
    """Diagnostic: a bounded wait on a barrier nothing completes must end in TIMEOUT."""
    _check("yoco_selftest_wait_timeout", lib.yoco_selftest_wait_timeout(
        _i32(err_word, "err_word"), int(limit_us), _stream(stream)))


def yoco_set_l2_window(base: Optional[torch.Tensor], nbytes: int, hit_ratio: float = 1.0,
                       stream=None) -> None:
    _check("yoco_set_l2_window", lib.yoco_set_l2_window(
        _stream(stream), None if base is None else base.data_ptr(), int(nbytes), float(hit_ratio)))


def yoco_version() -> int:
    return int(lib.yoco_version())


def yoco_last_cuda_error() -> int:
    return int(lib.yoco_last_cuda_error())


def yoco_last_cuda_error_string() -> str:
    return lib.yoco_last_cuda_error_string().decode()


def yoco_kv_append_e4m3(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                        v_cache: torch.Tensor, page_scales: torch.Tensor, block_table: torch.Tensor,
                        seq_lens: torch.Tensor, query_start_loc: torch.Tensor,
                        err_word: Optional[torch.Tensor] = None, stream=None) -> None:
    """Quantising append: bf16 ``k_new/v_new [T, H_kv, D]`` into one-byte pools
    ``[num_blocks, H_kv, bs, D]`` with float32 ``page_scales [num_blocks, H_kv, 4]``."""
    num_blocks, H_kv, bs, D = k_cache.shape
    assert v_cache.shape == k_cache.shape and k_new.shape == v_new.shape
    assert k_new.dtype == v_new.dtype == torch.bfloat16
    assert k_cache.element_size() == 1 and v_cache.element_size() == 1
    assert page_scales.dtype == torch.float32 and tuple(page_scales.shape) == (num_blocks, H_kv, 4)
    T = k_new.shape[0]
    assert k_new.shape[1:] == (H_kv, D)
    R = query_start_loc.shape[0] - 1
    _check("yoco_kv_append_e4m3", lib.yoco_kv_append_e4m3(
        _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(page_scales),
        _i32(block_table, "block_table"), block_table.shape[1], _i32(seq_lens, "seq_lens"),
        _i32(query_start_loc, "query_start_loc"), R, T, num_blocks, bs, H_kv, D,
        None if err_word is None else _i32(err_word, "err_word"), _stream(stream)))


def yoco_cross_attn_paged_e4m3(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                               page_scales: torch.Tensor, out: torch.Tensor,
                               block_table: torch.Tensor, seq_lens: torch.Tensor,
                               cross_query_start_loc: torch.Tensor, max_seq_len: int, scale: float,
                               workspace: Optional[torch.Tensor],
                               err_word: Optional[torch.Tensor] = None, stream=None,
                               max_rows: Optional[int] = None, flags: int = 0) -> None:
    """One layer over an e4m3 cache: bf16 ``q/out [max_rows, H_q, D]``."""
    num_blocks, H_kv, bs, D = k_cache.shape
    rows_cap, H_q, Dq = q.shape
    assert Dq == D and out.shape == q.shape and out.dtype == q.dtype == torch.bfloat16
    assert k_cache.element_size() == 1 and v_cache.shape == k_cache.shape
    assert page_scales.dtype == torch.float32 and tuple(page_scales.shape) == (num_blocks, H_kv, 4)
    R = cross_query_start_loc.shape[0] - 1
    max_rows = rows_cap if max_rows is None else max_rows
    assert max_rows <= rows_cap
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("yoco_cross_attn_paged_e4m3", lib.yoco_cross_attn_paged_e4m3(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_scales), _ptr(out),
        _i32(block_table, "block_table"), block_table.shape[1], _i32(seq_lens, "seq_lens"),
        _i32(cross_query_start_loc, "cross_query_start_loc"), R, max_rows, int(max_seq_len), H_q,
        H_kv, D, bs, num_blocks, float(scale), int(flags), _ptr(workspace), ws_bytes,
        None if err_word is None else _i32(err_word, "err_word"), _stream(stream)))


def yoco_cross_decode_step(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                           k_cache: torch.Tensor, v_cache: torch.Tensor,
                           page_scales: Optional[torch.Tensor], out: torch.Tensor,
                           block_table: torch.Tensor, seq_lens: torch.Tensor,
                           query_start_loc: torch.Tensor, max_seq_len: int, scale: float,
                           workspace: Optional[torch.Tensor],
                           err_word: Optional[torch.Tensor] = None, stream=None,
                           flags: int = 0) -> None:
    """Decode step: append ``k_new/v_new [R, H_kv, D]`` and attend layer ``q [R, H_q, D]``."""
    num_blocks, H_kv, bs, D = k_cache.shape
    R, H_q, Dq = q.shape
    assert Dq == D and out.shape == q.shape and q.dtype == torch.bfloat16
    assert k_new.shape == v_new.shape == (R, H_kv, D) and k_new.dtype == torch.bfloat16
    assert query_start_loc.shape[0] == R + 1
    e4m3 = k_cache.element_size() == 1
    if e4m3:
        assert page_scales is not None and page_scales.dtype == torch.float32
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("yoco_cross_decode_step", lib.yoco_cross_decode_step(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
        _ptr(page_scales) if e4m3 else None, _ptr(out), _i32(block_table, "block_table"),
        block_table.shape[1], _i32(seq_lens, "seq_lens"),
        _i32(query_start_loc, "query_start_loc"), R, int(max_seq_len), H_q, H_kv, D, bs,
        num_blocks, float(scale), YOCO_E4M3 if e4m3 else YOCO_BF16, int(flags), _ptr(workspace),
        ws_bytes, None if err_word is None else _i32(err_word, "err_word"), _stream(stream)))

