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
    assert call(flags=0x10) == 1    # unknown flag bit
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


def test_e4m3_host_validation(lib_path):
    from yoco_shared_kv_gb300 import _native as N
    L = N.lib
    fake = 1 << 20  # never dereferenced: every call below returns before a launch

    def attn(**kw):
        a = dict(hq=8, hkv=2, d=256, bs=16, sc=fake, flags=0)
        a.update(kw)
        return L.yoco_cross_attn_paged_e4m3(fake, fake, fake, a["sc"], fake, fake, 4, fake, fake,
                                            1, 1, 64, a["hq"], a["hkv"], a["d"], a["bs"], 100,
                                            0.0625, a["flags"], None, 0, None, None)
    assert attn(d=64) == N.YOCO_ERR_UNSUPPORTED     # e4m3 pages need 128-byte rows
    assert attn(bs=8) == N.YOCO_ERR_UNSUPPORTED
    assert attn(sc=None) == N.YOCO_ERR_INVALID_ARG  # scale records are required
    assert attn(sc=fake + 8) == N.YOCO_ERR_INVALID_ARG  # 16-byte records, 16-byte aligned
    assert attn(flags=0x10) == N.YOCO_ERR_INVALID_ARG  # unknown flag bit
    assert attn() == N.YOCO_ERR_WORKSPACE           # no workspace given
    # the bf16 entry refuses the e4m3 dtype
    assert L.yoco_cross_attn_paged(fake, fake, fake, fake, fake, 4, fake, fake, 1, 1, 64, 8, 2,
                                   256, 16, 100, 0.0625, N.YOCO_E4M3, 0, None, 0, None,
                                   None) == N.YOCO_ERR_UNSUPPORTED

    def app(**kw):
        a = dict(d=128, sc=fake)
        a.update(kw)
        return L.yoco_kv_append_e4m3(fake, fake, fake, fake, a["sc"], fake, 4, fake, fake, 1, 1,
                                     100, 16, 2, a["d"], None, None)
    assert app(d=64) == N.YOCO_ERR_UNSUPPORTED
    assert app(sc=None) == N.YOCO_ERR_INVALID_ARG
    assert app(sc=fake + 4) == N.YOCO_ERR_INVALID_ARG


def test_e4m3_workspace_and_traffic(lib_path):
    from yoco_shared_kv_gb300 import _native as N
    import torch
    f8 = torch.float8_e4m3fn
    assert N.yoco_cross_attn_workspace_size(4, 8, 2, 64, 16, 4096, f8) == 0
    a = N.yoco_cross_attn_workspace_size(4, 8, 2, 256, 16, 4096, f8)
    b = N.yoco_cross_attn_workspace_size(64, 8, 2, 256, 16, 131072, f8)
    assert a == b > 0
    # one request, one row over 100 keys: K/V bytes halve, scale records are added
    tb, _ = N.yoco_cross_decoder_bytes([0, 1], None, [100], 1, 8, 2, 128, 16, torch.bfloat16)
    t8, _ = N.yoco_cross_decoder_bytes([0, 1], None, [100], 1, 8, 2, 128, 16, f8)
    pages = 7
    assert tb == 100 * 2 * 2 * 128 * 2 + 2 * 8 * 128 * 2 + 4 * pages * 2
    assert t8 == 100 * 2 * 2 * 128 * 1 + 2 * 8 * 128 * 2 + 20 * pages * 2


def test_fused_step_host_validation(lib_path):
    from yoco_shared_kv_gb300 import _native as N
    L = N.lib
    fake = 1 << 20  # never dereferenced: every call below returns before a launch

    def step(**kw):
        a = dict(kn=fake, dt=N.YOCO_BF16, flags=0, d=256)
        a.update(kw)
        return L.yoco_cross_decode_step(fake, a["kn"], fake, fake, fake, fake, fake, fake, 4,
                                        fake, fake, 1, 64, 8, 2, a["d"], 16, 100, 0.0625, a["dt"],
                                        a["flags"], None, 0, None, None)
    assert step(flags=N.YOCO_ATTN_REVERSE) == N.YOCO_ERR_INVALID_ARG  # the step walks forward
    assert step(dt=N.YOCO_F32) == N.YOCO_ERR_UNSUPPORTED
    assert step(kn=None) == N.YOCO_ERR_INVALID_ARG
    assert step(kn=fake + 8) == N.YOCO_ERR_INVALID_ARG
    assert step(d=96) == N.YOCO_ERR_UNSUPPORTED
    assert step() == N.YOCO_ERR_WORKSPACE  # every check passed, no workspace given
    # the allocation-free entry does not take the e4m3 cache
    assert L.yoco_cross_attn_paged_noalloc(fake, fake, fake, fake, fake, 4, fake, fake, 1, 1, 64,
                                           8, 2, 256, 16, 100, 0.0625, N.YOCO_E4M3, None,
                                           None) == N.YOCO_ERR_UNSUPPORTED


def test_append_host_validation(lib_path):
    """yoco_kv_append rejects bad arguments before any CUDA call (the pointers
    below are never dereferenced), and an empty batch is a no-op."""
    from yoco_shared_kv_gb300 import _native as N
    L = N.lib
    fake = 1 << 20

    def app(**kw):
        a = dict(kn=fake, kc=fake, maxb=4, R=1, T=1, nb=100, bs=16, hkv=2, d=128, dt=N.YOCO_BF16)
        a.update(kw)
        return L.yoco_kv_append(a["kn"], fake, a["kc"], fake, fake, a["maxb"], fake, fake, a["R"],
                                a["T"], a["nb"], a["bs"], a["hkv"], a["d"], a["dt"], None, None)
    assert app(dt=N.YOCO_E4M3) == N.YOCO_ERR_UNSUPPORTED  # the 8-bit cache has its own entry
    assert app(dt=7) == N.YOCO_ERR_UNSUPPORTED
    assert app(d=96) == N.YOCO_ERR_UNSUPPORTED
    assert app(bs=24) == N.YOCO_ERR_UNSUPPORTED
    assert app(R=-1) == N.YOCO_ERR_INVALID_ARG
    assert app(T=-1) == N.YOCO_ERR_INVALID_ARG
    assert app(nb=0) == N.YOCO_ERR_INVALID_ARG
    assert app(hkv=0) == N.YOCO_ERR_INVALID_ARG
    assert app(maxb=0) == N.YOCO_ERR_INVALID_ARG
    assert app(kn=None) == N.YOCO_ERR_INVALID_ARG
    assert app(kc=fake + 8) == N.YOCO_ERR_INVALID_ARG    # 16-byte vector stores need alignment
    assert app(T=0, kn=None, kc=None) == N.YOCO_OK       # nothing to append: no launch
    assert app(R=0, kn=None, kc=None) == N.YOCO_OK


def test_noalloc_and_l2_window_host_validation(lib_path):
    """The allocation-free entry refuses the 8-bit dtype and bounds its fixed
    array cannot hold, and the L2 window refuses a hit ratio above 1, all
    before any CUDA call (the pointers are never dereferenced)."""
    import torch
    from yoco_shared_kv_gb300 import _native as N
    L = N.lib
    fake = 1 << 20
    cap = N.yoco_cross_attn_noalloc_capacity()
    assert cap > 0

    def noalloc(dt, H_q=8, H_kv=2, D=256, bs=16, rows=4, ctx=4096):
        return L.yoco_cross_attn_paged_noalloc(fake, fake, fake, fake, fake, 4, fake, fake, 1, rows,
                                               ctx, H_q, H_kv, D, bs, 100, ctypes.c_float(0.0625),
                                               dt, None, None)
    assert noalloc(N.YOCO_E4M3) == N.YOCO_ERR_UNSUPPORTED
    assert noalloc(9) == N.YOCO_ERR_UNSUPPORTED
    # the fp32 path's split grid, at the row count that makes it largest (16 heads,
    # head_dim 256, long contexts), needs more scratch than the array holds
    def need(r):
        return N.yoco_cross_attn_workspace_size(r, 16, 2, 256, 16, 65536, torch.float32)
    rows = max(range(1, 2048), key=need)
    assert need(rows) > cap
    assert noalloc(N.YOCO_F32, H_q=16, H_kv=2, rows=rows, ctx=65536) == N.YOCO_ERR_WORKSPACE
    L.yoco_set_l2_window.restype = ctypes.c_int
    L.yoco_set_l2_window.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                     ctypes.c_float]
    assert L.yoco_set_l2_window(None, fake, 1 << 20, 1.5) == N.YOCO_ERR_INVALID_ARG
    assert L.yoco_set_l2_window(None, fake, 1 << 20, float("nan")) == N.YOCO_ERR_INVALID_ARG


def test_plan_host_validation(lib_path):
    """yoco_cross_attn_plan checks its arguments before any launch; the fp32
    path plans on the host and returns without one."""
    import torch
    from yoco_shared_kv_gb300 import _native as N
    L = N.lib
    fake = 1 << 20  # never dereferenced: every call below returns before a launch

    def plan(dt=N.YOCO_BF16, d=128, bs=32, flags=0, ws=fake, ws_bytes=None, bt=fake, hq=16, hkv=1):
        need = N.yoco_cross_attn_workspace_size(4, hq, hkv, d, bs, 4096,
                                                {N.YOCO_BF16: torch.bfloat16,
                                                 N.YOCO_F32: torch.float32}.get(dt, torch.uint8))
        return L.yoco_cross_attn_plan(bt, 128, fake, fake, 4, 4, 4096, hq, hkv, d, bs, 1000, dt,
                                      flags, ws, need if ws_bytes is None else ws_bytes, None, None)
    assert plan(flags=N.YOCO_ATTN_REVERSE) == N.YOCO_ERR_INVALID_ARG   # only OVERLAP is taken
    assert plan(flags=N.YOCO_ATTN_PLANNED) == N.YOCO_ERR_INVALID_ARG
    assert plan(bt=None) == N.YOCO_ERR_INVALID_ARG
    assert plan(ws=fake + 8) == N.YOCO_ERR_INVALID_ARG                # 16-byte aligned workspace
    assert plan(ws_bytes=16) == N.YOCO_ERR_WORKSPACE
    assert plan(ws=None) == N.YOCO_ERR_WORKSPACE
    assert plan(d=96) == N.YOCO_ERR_UNSUPPORTED
    assert plan(dt=N.YOCO_E4M3, d=64) == N.YOCO_ERR_UNSUPPORTED      # e4m3 pages need 128-byte rows
    assert plan(hq=17, hkv=1) == N.YOCO_ERR_UNSUPPORTED
    assert plan(dt=N.YOCO_F32, ws=None, ws_bytes=0, hq=8, hkv=2) == N.YOCO_OK  # no plan needed


def test_noalloc_array_holds_every_tensor_core_shape(lib_path):
    """The attention workspace of the bf16 and e4m3 paths does not depend on context
    length or row count, and for every supported bf16 head_dim, block size and group
    (one row per request or row groups, one warp per ring or warp pairs) it fits the
    allocation-free entry's fixed array."""
    import torch
    from yoco_shared_kv_gb300 import _native as N
    cap = N.yoco_cross_attn_noalloc_capacity()
    for dt in (torch.bfloat16, torch.float8_e4m3fn):
        for D in (64, 128, 256):
            if dt is torch.float8_e4m3fn and D == 64:
                continue  # e4m3 pages need 128-byte rows
            for bs in (16, 32):
                for G in (1, 2, 3, 4, 8, 12, 16):
                    need = N.yoco_cross_attn_workspace_size(64, G * 2, 2, D, bs, 1 << 20, dt)
                    assert need > 0, (dt, D, bs, G)
                    assert need == N.yoco_cross_attn_workspace_size(4096, G * 2, 2, D, bs, 512, dt)
                    if dt is torch.bfloat16:
                        assert need <= cap, (D, bs, G, need)
