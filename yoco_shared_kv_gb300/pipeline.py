"""One scheduling step of the cross-decoder hot path on the GPU.

``DeviceWorkload`` holds a workload's buffers in device memory (the paged
K^/V^ pools, metadata, per-layer queries and outputs) and runs the path:

    yoco_kv_append          (shared K^/V^ of the step's tokens, once)
    yoco_select_cross_rows  (rows entering the cross-decoder)
    yoco_cross_attn_paged   x layers (each layer's own queries, same cache)

as in "YOCO 论文与推理数据流详解" §13.4 (self-prefill, global-KV finalize,
cross-decode) and "You Only Cache Once, in vLLM" (cross-decoder batch =
one row per scheduled request). Only allocation and argument marshalling
happen here; every step of the path runs in the CUDA library.
"""
from __future__ import annotations

from typing import List, Optional

import numpy as np
import torch

from . import _native as N


def to_torch(arr: np.ndarray, dtype: str) -> torch.Tensor:
    """Storage-dtype numpy array -> CPU torch tensor sharing its bits."""
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32))


def torch_dtype(dtype: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]


class DeviceStep:
    """Device copies of one step's inputs, plus its outputs and scratch."""

    def __init__(self, wl, step, device, pin_host: bool = False, e4m3: bool = False):
        self.wl, self.step = wl, step
        dev = torch.device(device)
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32))  # noqa: E731
        host = {
            "qsl": i32(step.query_start_loc),
            "seq_lens": i32(step.seq_lens),
            "block_table": i32(step.block_table),
            "k_new": to_torch(step.k_new, wl.dtype),
            "v_new": to_torch(step.v_new, wl.dtype),
        }
        if step.rows_per_req is not None:
            host["rows_per_req"] = i32(step.rows_per_req)
        if step.q is not None:
            host["q"] = to_torch(step.q, wl.dtype)
        if pin_host:
            host = {k: v.pin_memory() for k, v in host.items()}
        self.host = host
        self.dev = {k: v.to(dev) for k, v in host.items()}
        R, T = step.num_reqs, step.num_tokens
        self.num_reqs, self.num_tokens = R, T
        self.max_seq_len = int(step.seq_lens.max()) if R else 1
        self.rows_upper = step.rows_upper
        self.row_indices = torch.zeros(max(T, 1), dtype=torch.int32, device=dev)
        self.cqsl = torch.zeros(R + 1, dtype=torch.int32, device=dev)
        self.num_rows = torch.zeros(1, dtype=torch.int32, device=dev)
        self.out = None
        self.workspace = None
        if step.q is not None:
            self.out = torch.empty_like(self.dev["q"])
            ws = N.yoco_cross_attn_workspace_size(
                max(self.rows_upper, 1), wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                wl.block_size, self.max_seq_len,
                torch.float8_e4m3fn if e4m3 else torch_dtype(wl.dtype))
            # all-ones bytes (NaN as fp32): the library must never read scratch it
            # did not write in the same call, and this makes such a read visible
            self.workspace = torch.full((max(ws, 16),), 255, dtype=torch.uint8, device=dev)

    def h2d(self, stream=None) -> int:
        """Re-copy the step's inputs from (pinned) host memory; returns bytes copied."""
        nbytes = 0
        for k, v in self.host.items():
            self.dev[k].copy_(v, non_blocking=True)
            nbytes += v.numel() * v.element_size()
        return nbytes


class DeviceWorkload:
    """``kv="e4m3"`` keeps the cache as e4m3 bytes with per-(page, kv head) scale
    records ``page_scales`` (float32 numpy ``[num_blocks, H_kv, 4]``); the
    workload's values must then be bf16."""

    def __init__(self, wl, device="cuda", pin_host: bool = False, sentinel: bool = True,
                 alternate="auto", kv: str = "native", page_scales=None):
        self.wl = wl
        self.device = torch.device(device)
        self.e4m3 = kv == "e4m3"
        if kv not in ("native", "e4m3"):
            raise ValueError(kv)
        tdt = torch_dtype(wl.dtype)
        shape = wl.pool_shape()
        self.page_scales = None
        if self.e4m3:
            if wl.dtype != "bf16":
                raise ValueError("the e4m3 cache takes bf16 values")
            if page_scales is None:
                raise ValueError("an e4m3 cache needs page_scales")
            self.page_scales = torch.from_numpy(
                np.ascontiguousarray(page_scales, dtype=np.float32)).to(self.device)
            fill = 0xFF if sentinel else 0
            self.k_cache = torch.full(shape, fill, dtype=torch.uint8, device=self.device)
            self.v_cache = torch.full(shape, fill, dtype=torch.uint8, device=self.device)
        elif sentinel:
            # all-ones bytes: NaN in both dtypes, so a stray read poisons the output
            self.k_cache = torch.full(shape, -1, dtype=torch.int16 if tdt == torch.bfloat16
                                      else torch.int32, device=self.device).view(tdt)
            self.v_cache = torch.full(shape, -1, dtype=torch.int16 if tdt == torch.bfloat16
                                      else torch.int32, device=self.device).view(tdt)
        else:
            self.k_cache = torch.empty(shape, dtype=tdt, device=self.device)
            self.v_cache = torch.empty(shape, dtype=tdt, device=self.device)
        self.err = torch.zeros(1, dtype=torch.int32, device=self.device)
        if alternate == "auto":
            # Reverse every other layer's page walk only when the cache does not
            # fit in L2; a cache that fits is served from L2 in any order.
            pool_bytes = 2 * self.k_cache.numel() * self.k_cache.element_size()
            l2 = torch.cuda.get_device_properties(self.device).L2_cache_size
            alternate = pool_bytes > l2
        self.alternate = bool(alternate)
        e8 = self.e4m3
        self.fill = DeviceStep(wl, wl.fill, device, pin_host, e8) if wl.fill is not None else None
        self.steps: List[DeviceStep] = [DeviceStep(wl, s, device, pin_host, e8) for s in wl.steps]

    # ------------------------------------------------------------------ calls

    def append(self, ds: DeviceStep, stream=None) -> None:
        d = ds.dev
        if self.e4m3:
            N.yoco_kv_append_e4m3(d["k_new"], d["v_new"], self.k_cache, self.v_cache,
                                  self.page_scales, d["block_table"], d["seq_lens"], d["qsl"],
                                  self.err, stream)
            return
        N.yoco_kv_append(d["k_new"], d["v_new"], self.k_cache, self.v_cache, d["block_table"],
                         d["seq_lens"], d["qsl"], self.err, stream)

    def select(self, ds: DeviceStep, stream=None) -> None:
        d = ds.dev
        N.yoco_select_cross_rows(d["qsl"], d.get("rows_per_req"), ds.row_indices, ds.cqsl,
                                 ds.num_rows, self.err, stream)

    def plan(self, ds: DeviceStep, stream=None, cq: Optional[torch.Tensor] = None) -> None:
        """The step's attention plan (once per step, after the selection): every layer of
        the step then reuses it (YOCO_ATTN_PLANNED)."""
        d = ds.dev
        wl = self.wl
        N.yoco_cross_attn_plan(d["block_table"], d["seq_lens"], ds.cqsl if cq is None else cq,
                               ds.max_seq_len, ds.out.shape[1], wl.num_q_heads, wl.num_kv_heads,
                               wl.head_dim, wl.block_size, self.k_cache.shape[0],
                               torch.float8_e4m3fn if self.e4m3 else torch_dtype(wl.dtype),
                               ds.workspace, self.err, stream)

    def attend(self, ds: DeviceStep, layer: int, stream=None, q: Optional[torch.Tensor] = None,
               out: Optional[torch.Tensor] = None, cq: Optional[torch.Tensor] = None,
               planned: bool = True) -> None:
        """One cross-decoder layer. Odd layers walk the pages last to first, so each
        layer starts on what the previous one left in L2 (when `alternate` is on).
        Layers after the first overlap their start with the previous layer's end:
        the kernel before them (the previous layer's merge) writes none of the
        metadata or cache they read early; the first layer follows the row
        selection, which writes cross_query_start_loc, so it does not."""
        d = ds.dev
        flags = N.YOCO_ATTN_REVERSE if (self.alternate and layer % 2 == 1) else 0
        if self.alternate:  # the next layer starts where this one ends: keep that in L2
            flags |= N.YOCO_ATTN_KEEP_TAIL
        if layer > 0:
            flags |= N.YOCO_ATTN_OVERLAP
        if planned:  # the step's plan (plan() or the fused step) is in the workspace
            flags |= N.YOCO_ATTN_PLANNED
        if self.e4m3:
            N.yoco_cross_attn_paged_e4m3(
                d["q"][layer] if q is None else q, self.k_cache, self.v_cache, self.page_scales,
                ds.out[layer] if out is None else out, d["block_table"], d["seq_lens"],
                ds.cqsl if cq is None else cq, ds.max_seq_len, self.wl.scale, ds.workspace,
                self.err, stream, flags=flags)
            return
        N.yoco_cross_attn_paged(d["q"][layer] if q is None else q, self.k_cache, self.v_cache,
                                ds.out[layer] if out is None else out, d["block_table"],
                                d["seq_lens"], ds.cqsl if cq is None else cq, ds.max_seq_len,
                                self.wl.scale, ds.workspace, self.err, stream, flags=flags)

    def decode_only(self, i: int) -> bool:
        """Every request of step i schedules one token and gets one cross row."""
        st = self.steps[i].step
        qsl = np.asarray(st.query_start_loc)
        rpr = st.rows_per_req
        return bool((np.diff(qsl) == 1).all() and (rpr is None or (np.asarray(rpr) == 1).all())
                    and self.wl.dtype == "bf16")

    def step_buffers(self, i: int, pin_host: bool = True) -> DeviceStep:
        """Another set of device buffers (inputs, outputs, scratch) for step i, so that
        one set's inputs can be copied in while a step runs on the other."""
        return DeviceStep(self.wl, self.wl.steps[i], self.device, pin_host, self.e4m3)

    def fused_step(self, i: int, stream=None, layers: Optional[int] = None) -> None:
        self.fused_step_on(self.steps[i], stream, layers)

    def fused_step_on(self, ds: DeviceStep, stream=None, layers: Optional[int] = None) -> None:
        """A decode step with the append fused into layer 0 (yoco_cross_decode_step),
        then every later layer; the row selection is the identity for decode."""
        d = ds.dev
        N.yoco_cross_decode_step(d["q"][0], d["k_new"], d["v_new"], self.k_cache, self.v_cache,
                                 self.page_scales, ds.out[0], d["block_table"], d["seq_lens"],
                                 d["qsl"], ds.max_seq_len, self.wl.scale, ds.workspace, self.err,
                                 stream, flags=N.YOCO_ATTN_KEEP_TAIL if self.alternate else 0)
        for layer in range(1, self.wl.layers if layers is None else layers):
            self.attend(ds, layer, stream, cq=d["qsl"])  # the step's plan made above

    def run_fill(self, stream=None) -> None:
        if self.fill is not None:
            self.append(self.fill, stream)

    def run_step(self, i: int, stream=None, layers: Optional[int] = None) -> None:
        self.run_step_on(self.steps[i], stream, layers)

    def run_step_on(self, ds: DeviceStep, stream=None, layers: Optional[int] = None) -> None:
        """append -> select -> plan -> every cross-decoder layer, all on one stream."""
        self.append(ds, stream)
        self.select(ds, stream)
        self.plan(ds, stream)
        for layer in range(self.wl.layers if layers is None else layers):
            self.attend(ds, layer, stream)

    def run_all(self, stream=None) -> None:
        self.run_fill(stream)
        for i in range(len(self.steps)):
            self.run_step(i, stream)

    def error_bits(self) -> int:
        return int(self.err.item())
