"""The C-ABI library builds, loads and exports every entry point its header declares.

Host-side only: the calls made here return on argument validation before
anything touches a GPU.
"""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "yoco_kv.h")


@pytest.fixture(scope="module")
def lib_path():
    from yoco_shared_kv_gb300 import build
    return build.build()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(yoco_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_path():
    names = _declared()
    for n in ("yoco_kv_append", "yoco_select_cross_rows", "yoco_cross_attn_paged",
              "yoco_cross_attn_workspace_size"):
        assert n in names


def test_library_exports_every_declared_symbol(lib_path):
    L = ctypes.CDLL(lib_path)
    missing = [n for n in _declared() if not hasattr(L, n)]
    assert not missing, missing


def test_binding_names_match_header(lib_path):
    from yoco_shared_kv_gb300 import _native as N
    for n in _declared():
        assert hasattr(N, n) or n in ("yoco_status_string",), n
        assert n in N.EXPORTED


def test_status_strings_and_version(lib_path):
    from yoco_shared_kv_gb300 import _native as N
    assert N.status_name(0) == "ok"
    assert "workspace" in N.status_name(3)
    assert N.yoco_version() == 100
    assert N.yoco_last_cuda_error() == 0  # nothing has failed on this thread


def test_host_validation_rejects_before_launch(lib_path):
    L = ctypes.CDLL(lib_path)
    L.yoco_cross_attn_paged.restype = ctypes.c_int
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    L.yoco_cross_attn_paged.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32,
                                        i32, i32, i32, ctypes.c_float, ctypes.c_int,
                                        ctypes.c_uint32, vp, ctypes.c_size_t, vp, vp]
    args = dict(hq=8, hkv=2, d=256, bs=16, dt=1)

    def call(**kw):
        a = {**args, **kw}
        return L.yoco_cross_attn_paged(None, None, None, None, None, 4, None, None, 1, 1, 64,
                                       a["hq"], a["hkv"], a["d"], a["bs"], 100, 0.0625, a["dt"],
                                       a.get("flags", 0), None, 0, None, None)
    assert call(d=96) == 2          # unsupported head_dim
    assert call(bs=8) == 2          # unsupported block size
    assert call(hq=7) == 1          # H_q not a multiple of H_kv
    assert call(hq=34, hkv=2) == 2  # group of 17
    assert call(dt=5) == 2          # unknown dtype
    assert call() == 1              # null pointers
    assert call(flags=0x4) == 1     # unknown flag bit
    L.yoco_select_cross_rows.restype = ctypes.c_int
    L.yoco_select_cross_rows.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp]
    assert L.yoco_select_cross_rows(None, None, -1, None, None, None, None, None) == 1
    assert L.yoco_select_cross_rows(None, None, 3, None, None, None, None, None) == 1


def test_workspace_sizes(lib_path):
    from yoco_shared_kv_gb300 import _native as N
    import torch
    # fp32 split-KV path: partials grow with the longest context
    small = N.yoco_cross_attn_workspace_size(4, 16, 1, 128, 32, 4096, torch.float32)
    big = N.yoco_cross_attn_workspace_size(4, 16, 1, 128, 32, 131072, torch.float32)
    assert big > small >= 0
    # bf16 persistent path: two partials per worker, independent of context length
    a = N.yoco_cross_attn_workspace_size(4, 16, 1, 128, 32, 4096, torch.bfloat16)
    b = N.yoco_cross_attn_workspace_size(64, 16, 1, 128, 32, 131072, torch.bfloat16)
    assert a == b > 0
    assert N.yoco_cross_attn_workspace_size(4, 16, 1, 96, 32, 4096, torch.bfloat16) == 0
