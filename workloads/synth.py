"""Seeded synthetic inputs for the YOCO cross-decoder hot path.

This module only *generates inputs*: request lengths, physical page
permutations, block tables and N(0,1) values for the shared K^/V^ and for
the per-layer cross-decoder queries. It holds none of the method's
arithmetic (no slot computation, no row selection, no attention); both the
CUDA path and the CPU oracle consume what it produces.

Shapes follow the pages' problem statement:

* "You Only Cache Once, in vLLM", section "Implementation in vLLM": requests
  are batched with prefill and decode tokens mixed; ``query_start_loc`` holds
  exclusive offsets of each request's scheduled tokens and ``seq_lens`` the
  tokens in cache after this step (its worked example: qsl [0,15,20,28],
  seq_lens [41,31,40]). The R1/R2 three-step schedule of the same section is
  the ``toy`` workload.
* "KV cache memory systems", section "Contiguous allocation wastes capacity":
  logical token blocks map through a block table to non-contiguous physical
  pages; section "Prefix caching needs identity rules": completed prefix
  blocks are shared by reference between requests.

Value recipe: ``numpy.random.default_rng`` streams derived from one integer
seed; N(0,1) float32 samples, rounded to bfloat16 (round-to-nearest-even)
where the workload is bf16. A bf16 array is stored as its uint16 bit
pattern so that both consumers read the very same bits.
"""
from __future__ import annotations

import dataclasses
import zlib
from typing import List, Optional, Sequence, Tuple

import numpy as np

# Byte pattern that fills every pool slot before any append: an all-ones
# pattern is a NaN in both f32 and bf16, so a read of a slot that was never
# written poisons the result instead of passing silently.
SENTINEL_BYTE = 0xFF

DTYPES = ("f32", "bf16")


def elem_bytes(dtype: str) -> int:
    return {"f32": 4, "bf16": 2}[dtype]


def storage_np_dtype(dtype: str):
    return {"f32": np.float32, "bf16": np.uint16}[dtype]


def _f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 samples to bfloat16 (nearest, ties to even); returns uint16 bits.

    Inputs are finite N(0,1) samples, so the NaN/Inf branches of a general
    converter are not needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def _normal(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if dtype == "bf16":
        return _f32_to_bf16_bits(x)
    return x


@dataclasses.dataclass
class Step:
    """One scheduling step: a batch of requests with their scheduled tokens.

    ``req_ids[b]`` is the workload request held by batch entry ``b``.
    ``k_new``/``v_new`` are ``[T, H_kv, D]`` in batch-token order (storage
    dtype), ``q`` is ``[layers, rows_upper, H_q, D]`` with one query row slot
    per cross-decoder row the generator intends to ask for (``rows_per_req``
    entries, default one per request with scheduled tokens).
    """

    req_ids: List[int]
    query_start_loc: np.ndarray  # int32 [R+1]
    seq_lens: np.ndarray  # int32 [R]
    block_table: np.ndarray  # int32 [R, max_blocks]
    rows_per_req: Optional[np.ndarray]  # int32 [R] or None (= one row each)
    k_new: np.ndarray
    v_new: np.ndarray
    q: Optional[np.ndarray]  # [layers, rows_upper, H_q, D]; None for an append-only step

    @property
    def num_reqs(self) -> int:
        return len(self.req_ids)

    @property
    def num_tokens(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def rows_upper(self) -> int:
        return 0 if self.q is None else int(self.q.shape[1])


@dataclasses.dataclass
class Workload:
    name: str
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    layers: int
    scale: float
    max_blocks_per_req: int
    # request r owns logical blocks -> physical pages req_pages[r]
    req_pages: List[np.ndarray]
    # per-request token values: K/V = concat(prefix part, private part)
    prefix_len: int
    prefix_k: Optional[np.ndarray]
    prefix_v: Optional[np.ndarray]
    private_k: List[np.ndarray]
    private_v: List[np.ndarray]
    fill: Optional[Step]  # append-only step that writes pre-existing context
    steps: List[Step]
    description: str = ""

    @property
    def num_reqs_total(self) -> int:
        return len(self.req_pages)

    def request_kv(self, r: int) -> Tuple[np.ndarray, np.ndarray]:
        """Full contiguous ``[len, H_kv, D]`` K/V of request ``r`` (storage dtype)."""
        if self.prefix_len and r in self._prefix_users():
            k = np.concatenate([self.prefix_k, self.private_k[r]], axis=0)
            v = np.concatenate([self.prefix_v, self.private_v[r]], axis=0)
            return k, v
        return self.private_k[r], self.private_v[r]

    def _prefix_users(self):
        return range(self.num_reqs_total) if self.prefix_len else ()

    def kv_bytes_per_token(self) -> int:
        return 2 * self.num_kv_heads * self.head_dim * elem_bytes(self.dtype)

    def pool_shape(self) -> Tuple[int, int, int, int]:
        return (self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim)

    def empty_pool(self) -> np.ndarray:
        """A pool filled with the sentinel pattern (storage dtype)."""
        nbytes = int(np.prod(self.pool_shape())) * elem_bytes(self.dtype)
        raw = np.full(nbytes, SENTINEL_BYTE, dtype=np.uint8)
        return raw.view(storage_np_dtype(self.dtype)).reshape(self.pool_shape())


def _assemble_step(wl: Workload, entries: Sequence[Tuple[int, int, int]],
                   rows_per_req: Optional[Sequence[int]], rng_q: Optional[np.random.Generator],
                   with_q: bool) -> Step:
    """Build a batch from ``(request, seq_len, q_len)`` entries.

    The scheduled tokens of a request are the last ``q_len`` of its first
    ``seq_len`` tokens (the pages' worked example: 15 scheduled tokens of a
    request whose cache holds 41 after the step).
    """
    R = len(entries)
    qsl = np.zeros(R + 1, dtype=np.int32)
    seq = np.zeros(R, dtype=np.int32)
    bt = np.zeros((R, wl.max_blocks_per_req), dtype=np.int32)
    ks, vs = [], []
    for b, (r, s_len, q_len) in enumerate(entries):
        qsl[b + 1] = qsl[b] + q_len
        seq[b] = s_len
        pages = wl.req_pages[r]
        bt[b, : len(pages)] = pages
        k, v = wl.request_kv(r)
        ks.append(k[s_len - q_len:s_len])
        vs.append(v[s_len - q_len:s_len])
    shp = (0, wl.num_kv_heads, wl.head_dim)
    sdt = storage_np_dtype(wl.dtype)
    k_new = np.ascontiguousarray(np.concatenate(ks, axis=0)) if ks else np.zeros(shp, sdt)
    v_new = np.ascontiguousarray(np.concatenate(vs, axis=0)) if vs else np.zeros(shp, sdt)
    rpr = None if rows_per_req is None else np.asarray(rows_per_req, dtype=np.int32)
    q = None
    if with_q:
        # The generator only asks for rows a request actually has scheduled
        # tokens for, so the row count is known here without any selection.
        if rpr is None:
            assert all(q_len >= 1 for (_, _, q_len) in entries)
            rows_upper = R
        else:
            assert all(0 <= int(x) <= e[2] for x, e in zip(rpr, entries))
            rows_upper = int(rpr.sum())
        q = _normal(rng_q, (wl.layers, rows_upper, wl.num_q_heads, wl.head_dim), wl.dtype)
    return Step(req_ids=[e[0] for e in entries], query_start_loc=qsl, seq_lens=seq,
                block_table=bt, rows_per_req=rpr, k_new=k_new, v_new=v_new, q=q)


def _allocate_pages(rng: np.random.Generator, blocks_needed: Sequence[int], pool_factor: float,
                    min_pool: int = 0, shared_prefix_blocks: int = 0):
    """Random physical placement: a permuted pool sized ``pool_factor`` x the blocks in use.

    With ``shared_prefix_blocks`` > 0 the first that many logical blocks of
    every request reference the same physical pages (a refcounted prefix);
    ``blocks_needed`` then counts each request's *private* blocks only.
    """
    used = shared_prefix_blocks + int(sum(blocks_needed))
    num_blocks = max(int(np.ceil(pool_factor * used)), used, min_pool)
    perm = rng.permutation(num_blocks).astype(np.int32)
    prefix = perm[:shared_prefix_blocks]
    cur = shared_prefix_blocks
    pages = []
    for nb in blocks_needed:
        pages.append(np.concatenate([prefix, perm[cur:cur + nb]]).astype(np.int32))
        cur += nb
    return num_blocks, pages


def _make(name, *, dtype, H_q, H_kv, D, bs, layers, seed, full_lens, step_entries,
          rows_per_req=None, pool_factor=1.2, min_pool=0, prefix_len=0, description=""):
    """Generic builder: requests of final length ``full_lens``; one timed step.

    ``step_entries`` = list of ``(request, seq_len, q_len)`` for the step.
    Context tokens ``[0, seq_len - q_len)`` are written by an append-only
    ``fill`` step before the timed step (the shared prefix only once, by the
    first request that holds it).
    """
    assert dtype in DTYPES
    rng_struct = np.random.default_rng([seed, 0])
    rng_kv = np.random.default_rng([seed, 1])
    rng_q = np.random.default_rng([seed, 2])
    assert prefix_len % bs == 0
    pblocks = prefix_len // bs
    private_blocks = [-(-(n - prefix_len) // bs) for n in full_lens]
    num_blocks, pages = _allocate_pages(rng_struct, private_blocks, pool_factor, min_pool, pblocks)
    max_blocks = max(len(p) for p in pages) if pages else 1
    prefix_k = prefix_v = None
    if prefix_len:
        prefix_k = _normal(rng_kv, (prefix_len, H_kv, D), dtype)
        prefix_v = _normal(rng_kv, (prefix_len, H_kv, D), dtype)
    priv_lens = [n - prefix_len for n in full_lens]
    tot = int(sum(priv_lens))
    allk = _normal(rng_kv, (tot, H_kv, D), dtype)
    allv = _normal(rng_kv, (tot, H_kv, D), dtype)
    offs = np.concatenate([[0], np.cumsum(priv_lens)]).astype(np.int64)
    private_k = [allk[offs[i]:offs[i + 1]] for i in range(len(full_lens))]
    private_v = [allv[offs[i]:offs[i + 1]] for i in range(len(full_lens))]
    wl = Workload(name=name, dtype=dtype, num_q_heads=H_q, num_kv_heads=H_kv, head_dim=D,
                  block_size=bs, num_blocks=num_blocks, layers=layers, scale=1.0 / np.sqrt(D),
                  max_blocks_per_req=max_blocks, req_pages=pages, prefix_len=prefix_len,
                  prefix_k=prefix_k, prefix_v=prefix_v, private_k=private_k, private_v=private_v,
                  fill=None, steps=[], description=description)
    fill_entries = []
    prefix_written = False
    for (r, s_len, q_len) in step_entries:
        ctx = s_len - q_len
        start = 0
        if prefix_len and ctx > 0:
            if prefix_written:
                start = min(prefix_len, ctx)
            prefix_written = prefix_written or ctx >= prefix_len
        if ctx - start > 0:
            fill_entries.append((r, ctx, ctx - start))
    if fill_entries:
        wl.fill = _assemble_step(wl, fill_entries, None, None, with_q=False)
    wl.steps = [_assemble_step(wl, step_entries, rows_per_req, rng_q, with_q=True)]
    return wl


# ---------------------------------------------------------------- workloads


def toy_r1r2(seed: int = 1000) -> Workload:
    """R1/R2 mixed batch of "You Only Cache Once, in vLLM" (Implementation in vLLM).

    R1: 6-token prompt, R2: 2-token prompt; three scheduling steps
    (R1 prefill; R1 decode + R2 prefill; both decode). fp32, H_q=4, H_kv=1,
    head_dim=64, block_size=16, a pool of 8 physical pages in random order,
    8 cross-decoder layers with fresh N(0,1) queries, scale 1/sqrt(64).
    """
    dtype, H_q, H_kv, D, bs, layers = "f32", 4, 1, 64, 16, 8
    rng_struct = np.random.default_rng([seed, 0])
    rng_kv = np.random.default_rng([seed, 1])
    rng_q = np.random.default_rng([seed, 2])
    perm = rng_struct.permutation(8).astype(np.int32)
    pages = [perm[0:1].copy(), perm[1:2].copy()]
    full = [8, 3]
    private_k = [_normal(rng_kv, (n, H_kv, D), dtype) for n in full]
    private_v = [_normal(rng_kv, (n, H_kv, D), dtype) for n in full]
    wl = Workload(name="toy_r1r2_f32", dtype=dtype, num_q_heads=H_q, num_kv_heads=H_kv,
                  head_dim=D, block_size=bs, num_blocks=8, layers=layers, scale=1.0 / np.sqrt(D),
                  max_blocks_per_req=1, req_pages=pages, prefix_len=0, prefix_k=None,
                  prefix_v=None, private_k=private_k, private_v=private_v, fill=None, steps=[],
                  description="R1/R2 three-step toy schedule, fp32")
    schedule = [
        [(0, 6, 6)],            # step 0: R1 prefill, tokens 0..5
        [(0, 7, 1), (1, 2, 2)],  # step 1: R1 decode (token 6) + R2 prefill (tokens 0..1)
        [(0, 8, 1), (1, 3, 1)],  # step 2: both decode
    ]
    wl.steps = [_assemble_step(wl, s, None, rng_q, with_q=True) for s in schedule]
    return wl


def pure_decode(seed: int = 1001, num_reqs: int = 64, ctx_lo: int = 1024, ctx_hi: int = 8192,
                H_q: int = 8, H_kv: int = 2, D: int = 256, bs: int = 16, layers: int = 10,
                dtype: str = "bf16", explicit_lens: Optional[Sequence[int]] = None) -> Workload:
    """Pure decode: one new token per request; context lengths uniform in [lo, hi]."""
    rng = np.random.default_rng([seed, 3])
    lens = list(explicit_lens) if explicit_lens is not None else \
        [int(x) for x in rng.integers(ctx_lo, ctx_hi, size=num_reqs, endpoint=True)]
    entries = [(r, n, 1) for r, n in enumerate(lens)]
    return _make(f"pure_decode_{dtype}", dtype=dtype, H_q=H_q, H_kv=H_kv, D=D, bs=bs,
                 layers=layers, seed=seed, full_lens=lens, step_entries=entries,
                 description=f"pure decode: {len(lens)} requests, ctx U[{ctx_lo},{ctx_hi}]")


def mixed_step(seed: int = 1002, n_decode: int = 16, dec_lo: int = 2048, dec_hi: int = 16384,
               n_prefill: int = 4, pre_lo: int = 1024, pre_hi: int = 8192, H_q: int = 8,
               H_kv: int = 2, D: int = 256, bs: int = 16, layers: int = 10,
               dtype: str = "bf16", rows_per_req: Optional[Sequence[int]] = None) -> Workload:
    """Continuous-batching step: decoding requests first, then prefilling prompts.

    Every prompt token's K^/V^ is appended in the step; only the decode rows
    and the last prompt row of each prefill enter the cross-decoder.
    """
    rng = np.random.default_rng([seed, 3])
    dec = [int(x) for x in rng.integers(dec_lo, dec_hi, size=n_decode, endpoint=True)]
    pre = [int(x) for x in rng.integers(pre_lo, pre_hi, size=n_prefill, endpoint=True)]
    lens = dec + pre
    entries = [(r, n, 1) for r, n in enumerate(dec)] + \
              [(n_decode + i, n, n) for i, n in enumerate(pre)]
    return _make(f"mixed_{dtype}", dtype=dtype, H_q=H_q, H_kv=H_kv, D=D, bs=bs, layers=layers,
                 seed=seed, full_lens=lens, step_entries=entries, rows_per_req=rows_per_req,
                 description=f"mixed: {n_decode} decode ctx U[{dec_lo},{dec_hi}] + "
                             f"{n_prefill} prefill U[{pre_lo},{pre_hi}]")


def long_context(seed: int = 1003, num_reqs: int = 4, ctx: int = 131072, H_q: int = 16,
                 H_kv: int = 1, D: int = 128, bs: int = 32, layers: int = 12,
                 dtype: str = "bf16") -> Workload:
    """Long-context MQA decode: equal long contexts, permuted pages."""
    lens = [ctx] * num_reqs
    entries = [(r, n, 1) for r, n in enumerate(lens)]
    return _make(f"long_context_{dtype}", dtype=dtype, H_q=H_q, H_kv=H_kv, D=D, bs=bs,
                 layers=layers, seed=seed, full_lens=lens, step_entries=entries,
                 description=f"long-context decode: {num_reqs} x {ctx} tokens, MQA")


def shared_prefix(seed: int = 1004, num_reqs: int = 256, prefix_len: int = 4096, tail_lo: int = 64,
                  tail_hi: int = 512, H_q: int = 8, H_kv: int = 2, D: int = 128, bs: int = 32,
                  layers: int = 10, dtype: str = "bf16") -> Workload:
    """Decode batch whose block tables all reference one shared prefix plus private tails."""
    rng = np.random.default_rng([seed, 3])
    tails = [int(x) for x in rng.integers(tail_lo, tail_hi, size=num_reqs, endpoint=True)]
    lens = [prefix_len + t for t in tails]
    entries = [(r, n, 1) for r, n in enumerate(lens)]
    return _make(f"shared_prefix_{dtype}", dtype=dtype, H_q=H_q, H_kv=H_kv, D=D, bs=bs,
                 layers=layers, seed=seed, full_lens=lens, step_entries=entries,
                 prefix_len=prefix_len,
                 description=f"shared prefix {prefix_len} + tails U[{tail_lo},{tail_hi}] x {num_reqs}")


def spec_decode(seed: int = 1006, num_reqs: int = 64, ctx_lo: int = 1024, ctx_hi: int = 8192,
                draft: int = 4, H_q: int = 8, H_kv: int = 2, D: int = 256, bs: int = 16,
                layers: int = 10, dtype: str = "bf16") -> Workload:
    """Speculative verification at the pure-decode shapes: every request schedules
    `draft` tokens (the draft to verify) and asks for all of them as cross rows
    ("You Only Cache Once, in vLLM": the metadata builder gives a request several
    rows); contexts uniform in [lo, hi] before the draft."""
    rng = np.random.default_rng([seed, 3])
    ctx = [int(x) for x in rng.integers(ctx_lo, ctx_hi, size=num_reqs, endpoint=True)]
    lens = [c + draft for c in ctx]
    entries = [(r, n, draft) for r, n in enumerate(lens)]
    return _make(f"spec_decode_{dtype}", dtype=dtype, H_q=H_q, H_kv=H_kv, D=D, bs=bs,
                 layers=layers, seed=seed, full_lens=lens, step_entries=entries,
                 rows_per_req=[draft] * num_reqs,
                 description=f"speculative verification: {num_reqs} requests x {draft} rows, "
                             f"ctx U[{ctx_lo},{ctx_hi}]")


def chunked_prefill_spec(seed: int = 1005, H_q: int = 8, H_kv: int = 2, D: int = 128, bs: int = 16,
                         layers: int = 3, dtype: str = "bf16") -> Workload:
    """Three scheduling steps mixing a chunked prefill, a decode and a speculative decode.

    Request A: a 100-token prompt prefilled in chunks of 40, 40 and 20; only the
    last chunk's last token enters the cross-decoder (rows_per_req 0, 0, 1: the
    vLLM post notes that intermediate chunks could be skipped). Request B
    decodes one token per step after a 300-token context. Request C verifies 3
    draft tokens per step after a 200-token context and asks for all 3 trailing
    rows (the metadata builder's example gives a request several rows).
    """
    rng_struct = np.random.default_rng([seed, 0])
    rng_kv = np.random.default_rng([seed, 1])
    rng_q = np.random.default_rng([seed, 2])
    full = [100, 303, 209]
    blocks = [-(-n // bs) for n in full]
    num_blocks, pages = _allocate_pages(rng_struct, blocks, 1.2)
    private_k = [_normal(rng_kv, (n, H_kv, D), dtype) for n in full]
    private_v = [_normal(rng_kv, (n, H_kv, D), dtype) for n in full]
    wl = Workload(name=f"chunked_prefill_spec_{dtype}", dtype=dtype, num_q_heads=H_q,
                  num_kv_heads=H_kv, head_dim=D, block_size=bs, num_blocks=num_blocks,
                  layers=layers, scale=1.0 / np.sqrt(D), max_blocks_per_req=max(blocks),
                  req_pages=pages, prefix_len=0, prefix_k=None, prefix_v=None,
                  private_k=private_k, private_v=private_v, fill=None, steps=[],
                  description="chunked prefill (40/40/20) + decode + 3-token speculative decode")
    schedule = [
        ([(0, 40, 40), (1, 301, 1), (2, 203, 3)], [0, 1, 3]),
        ([(0, 80, 40), (1, 302, 1), (2, 206, 3)], [0, 1, 3]),
        ([(0, 100, 20), (1, 303, 1), (2, 209, 3)], [1, 1, 3]),
    ]
    wl.fill = _assemble_step(wl, [(1, 300, 300), (2, 200, 200)], None, None, with_q=False)
    wl.steps = [_assemble_step(wl, e, rpr, rng_q, with_q=True) for e, rpr in schedule]
    return wl


# The five workloads at full size, indexed as they are listed in the
# problem statement (0 = toy ... 4 = shared prefix).
FULL = {
    0: lambda: toy_r1r2(1000),
    1: lambda: pure_decode(1001),
    2: lambda: mixed_step(1002),
    3: lambda: long_context(1003),
    4: lambda: shared_prefix(1004),
}

# Scaled-down versions that still span several pages, splits and a ragged
# tail, small enough for the oracle to check every output in seconds.
SMALL = {
    0: lambda: toy_r1r2(1000),
    1: lambda: pure_decode(2001, num_reqs=6, ctx_lo=1, ctx_hi=1200,
                           explicit_lens=[1, 16, 17, 700, 1199, 333]),
    2: lambda: mixed_step(2002, n_decode=3, dec_lo=100, dec_hi=900, n_prefill=2, pre_lo=20,
                          pre_hi=300),
    3: lambda: long_context(2003, num_reqs=2, ctx=3000, layers=3),
    4: lambda: shared_prefix(2004, num_reqs=5, prefix_len=256, tail_lo=1, tail_hi=70, layers=3),
}

# Beyond the five: speculative verification (several cross rows per request)
# at the pure-decode shapes, full size and scaled down.
MULTI_ROW_FULL = lambda: spec_decode(1006)  # noqa: E731
MULTI_ROW_SMALL = lambda: spec_decode(2006, num_reqs=5, ctx_lo=1, ctx_hi=900, layers=2)  # noqa: E731


def page_scales(wl: Workload, lo: float = 3.5, hi: float = 5.0) -> np.ndarray:
    """Scale records of an 8-bit (e4m3) cache: float32 ``[num_blocks, H_kv, 4]``
    holding (k_scale, v_scale, 0, 0) per physical page and kv head.

    Recipe: each scale is A / 448 with A ~ U[lo, hi), i.e. the page-head can
    hold values up to A before saturating; K and V draw independently. For the
    N(0,1) values of these workloads that saturates a few values in 10^4 to
    10^6. Seeded by the workload's name and pool size.
    """
    rng = np.random.default_rng([zlib.crc32(wl.name.encode()), wl.num_blocks, 4])
    rec = np.zeros((wl.num_blocks, wl.num_kv_heads, 4), dtype=np.float32)
    rec[..., 0] = (rng.uniform(lo, hi, size=rec.shape[:2]) / 448.0).astype(np.float32)
    rec[..., 1] = (rng.uniform(lo, hi, size=rec.shape[:2]) / 448.0).astype(np.float32)
    return rec


def describe(wl: Workload) -> dict:
    st = wl.steps[-1]
    return {
        "workload": wl.name, "dtype": wl.dtype, "H_q": wl.num_q_heads, "H_kv": wl.num_kv_heads,
        "head_dim": wl.head_dim, "block_size": wl.block_size, "num_blocks": wl.num_blocks,
        "layers": wl.layers, "num_reqs": st.num_reqs, "num_tokens": st.num_tokens,
        "rows": st.rows_upper,
    }
