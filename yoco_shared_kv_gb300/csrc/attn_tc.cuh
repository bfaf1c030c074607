// Tensor-core cross-decoder attention: persistent and page-balanced
// (internal header: the kernel templates, instantiated by attn_tc.cu for a
// bf16 cache and by attn_tc_e4m3.cu for an e4m3 cache).
//
// "KV cache memory systems", "Cache contents": out = softmax(q K^T/sqrt(d_h)) V
// over the cached keys; "Contiguous allocation wastes capacity": every
// logical block is resolved through the block table. "YOCO 论文与推理数据流
// 详解" §10.4/§11: each cross-decoder layer streams the whole shared cache
// once with its own queries, so a layer is an HBM stream.
//
// Work decomposition. The unit of work is a page of one (cross row, kv head)
// segment. Segments are laid out in the order (row, kv head) and their pages
// form one flattened sequence of P pages. The grid has one CTA per SM; CTA c
// owns pages [P c / C, P (c+1) / C) and each of its workers owns an equal
// contiguous slice of that, streamed through the worker's own TMA ring. A
// worker is a warp, or (PR) a pair of warps that share the ring and split
// the group's 16 columns. Every worker therefore moves the same number of
// bytes, whatever the length mix, and the ring never drains between
// segments. Where each worker's slice starts is worked out once per step
// (attn_tc_plan) and read by every layer.
//   - A segment that lies inside one worker's slice is finished in registers
//     and written straight to `out`.
//   - A segment cut by a worker boundary leaves a partial (m, l, o) per piece;
//     at the end of the kernel the CTA combines the pieces of each segment
//     it holds, writing `out` when the CTA holds the whole segment and a
//     CTA-level partial otherwise.
//   - A segment cut by a CTA boundary is finished inside the same launch:
//     its CTAs meet at a counter, then each combines an equal share of the
//     segment's outputs from all their partials, in CTA order.
// Every combine runs in a fixed order that depends only on logical page
// indices, so the output is bit-identical under any physical page placement.
//
// Code that runs once per launch (the prologue and everything after the
// stream) is kept in rolled loops: it executes with a cold instruction
// cache, where each straight-line block costs instruction fetches from L2 or
// DRAM, so its size, more than its arithmetic, sets its time.
//
// Per page (one kv head, block_size tokens): K and V arrive by TMA as
// head_dim/64 tiles of [block_size x 128 B] with the 128-byte swizzle (so
// ldmatrix is conflict free); S^T = K Q^T and O^T += V^T P^T are m16n8k16
// bf16 mma.sync products with fp32 accumulators, the group's query heads on
// the N side; P moves from the accumulator layout to the B-operand layout
// with movmatrix. The online softmax works in the log2 domain.
#pragma once

#include "attn_common.cuh"

namespace yoco {
namespace {

// Warps per CTA and ring depth per warp for 16 KiB stages (compile-time
// tunables; the defaults fill 192 KiB of shared memory). Six warps of two
// stages keep as many bytes in flight as four of three, with half again as
// many warps to hide each page's chain of dependent steps. The warp count
// must be even.
#ifndef YOCO_TC_NW16
#define YOCO_TC_NW16 6
#endif
#ifndef YOCO_TC_ST16
#define YOCO_TC_ST16 2
#endif
// Two-tile walks as warp pairs, per head_dim (1 = on).
#ifndef YOCO_TC_PAIRS256
#define YOCO_TC_PAIRS256 1
#endif
#ifndef YOCO_TC_PAIRS128
#define YOCO_TC_PAIRS128 0
#endif
// e4m3 cache: warps per CTA and shared-memory bytes of the warps' rings
// (0 = derived from the piece sizes, below)
#ifndef YOCO_TC_F8_NW
#define YOCO_TC_F8_NW 0
#endif
#ifndef YOCO_TC_F8_RING
#define YOCO_TC_F8_RING 196608
#endif

// F8: the cache holds e4m3 bytes (one byte per element) instead of bf16.
// NT: 8-head tiles of a warp (1 for groups up to 8, else 2).
// PR: warp pairs (NT = 1): the two warps of a pair walk the same pages from
// one ring, each taking one of the group's two 8-head tiles, so a 16-column
// walk runs on twice the warps in the same shared memory.
template <int D, int BS, bool F8 = false, int NT = 2, bool PR = false>
struct TcShape {
    static_assert(!PR || NT == 1, "a warp of a pair takes one 8-head tile");
    static constexpr int ESZ = F8 ? 1 : 2;                // bytes per cached element
    static constexpr int PAGE_BYTES = BS * D * ESZ;       // K (or V) of one page, one kv head
    static constexpr int STAGE_BYTES = 2 * PAGE_BYTES;    // K + V
    static constexpr int NTG = PR ? 2 : NT;               // 8-head tiles of the group
    // a worker's (warp's, or pair's) two end-of-slice pieces at the largest group
    static constexpr int PIECE_PAIR = 2 * (8 * NTG * (D * 4 + 8) + 16);
    // the most workers (8, 4, 2) whose ring share holds two stages and the two pieces
    static constexpr int F8_FITS8 =
        PIECE_PAIR <= YOCO_TC_F8_RING / 8 && 2 * STAGE_BYTES <= YOCO_TC_F8_RING / 8;
    static constexpr int F8_FITS4 =
        PIECE_PAIR <= YOCO_TC_F8_RING / 4 && 2 * STAGE_BYTES <= YOCO_TC_F8_RING / 4;
    static constexpr int F8_NW =
        YOCO_TC_F8_NW > 0 ? YOCO_TC_F8_NW : (F8_FITS8 ? 8 : (F8_FITS4 ? 4 : 2));
    // Two 8-head tiles of one warp at head_dim 256 hold the queries in shared
    // memory (below): their kernels keep 4 warps x 3 stages whatever the
    // tunables say; so do the pair kernels (4 pairs x 3 stages).
    static constexpr bool QSM = D == 256 && NT == 2;
    // workers (each with its own ring and slice), and warps
    static constexpr int WK =
        F8 ? F8_NW
           : (STAGE_BYTES <= 8192 ? 8
                                  : (STAGE_BYTES <= 16384 ? ((QSM || PR) ? 4 : YOCO_TC_NW16) : 2));
    static constexpr int NW = PR ? 2 * WK : WK;
    // e4m3 pages are small: deepen the ring to keep ~192 KiB in flight per SM
    static constexpr int F8_STAGES = YOCO_TC_F8_RING / F8_NW / STAGE_BYTES;
    static constexpr int STAGES =
        F8 ? (F8_STAGES < 2 ? 2 : F8_STAGES)
           : (STAGE_BYTES == 16384 ? ((QSM || PR) ? 3 : YOCO_TC_ST16) : 3);
    static constexpr int SUBE = 128 / ESZ;  // elements per 128-byte row of a sub-tile
    static constexpr int KSUB = D / SUBE;   // 128-byte swizzled sub-tiles per row
    static constexpr int SUB_BYTES = BS * 128;
    static constexpr int MT = BS / 16;   // 16-token tiles per page
    static constexpr int KD = D / 16;    // 16-wide steps along head_dim
    // Two 8-head tiles at head_dim 256 would hold the queries in 64 registers
    // on top of the 128 of the output accumulators: there the queries of the
    // segment sit in shared memory instead (16 rows x D, 16-bit), read per
    // page with ldmatrix.
    static constexpr int Q_BYTES = QSM ? 16 * D * 2 : 0;  // per warp
    static constexpr int RING_BYTES = WK * STAGES * STAGE_BYTES;
    static constexpr int SMEM = RING_BYTES + NW * Q_BYTES + 1024;
    static_assert(SMEM <= 225 * 1024, "the rings must leave room for static shared memory");
};

// Byte offset of (token t, 16-byte chunk j of head-dim sub-tile c) in a
// 128B-swizzled page tile.
template <int BS>
__device__ __forceinline__ uint32_t swz(int c, int t, int j) {
    return static_cast<uint32_t>(c * (BS * 128) + t * 128 + ((j ^ (t & 7)) << 4));
}

// ------------------------------------------------------------- work order

__device__ __forceinline__ int32_t row_pages(int32_t kv_len, int32_t cap, int32_t bs) {
    if (kv_len <= 0) return 0;
    if (kv_len > cap) kv_len = cap;
    return (kv_len + bs - 1) / bs;
}

// Rows of a request are taken in groups of up to p.rg consecutive rows (below
// max_rows); a group's rows share one walk over the request's pages, up to the
// last row's causal end. Keys of the group's last row: row n of a request with
// k rows starting at c0 sees seq - k + (n - c0) + 1 keys.
__device__ __forceinline__ int32_t group_kv(int32_t seq, int32_t k, int32_t c0, int32_t n,
                                            int32_t nr) {
    return seq - k + (n + nr - c0);
}

// Pages (all kv heads) of request r's cross-row groups below max_rows.
__device__ __forceinline__ int64_t req_pages(const AttnParams& p, int32_t r, int32_t cap) {
    const int32_t c0 = __ldg(p.cqsl + r), c1 = __ldg(p.cqsl + r + 1);
    const int32_t k = c1 - c0, hi = min(c1, p.max_rows), seq = __ldg(p.seq_lens + r);
    int64_t s = 0;
    for (int32_t n = c0; n < hi; n += p.rg)
        s += row_pages(group_kv(seq, k, c0, n, min(p.rg, hi - n)), cap, p.block_size);
    return s * p.H_kv;
}

__device__ __forceinline__ int64_t warp_sum64(int64_t v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ int64_t warp_incl_scan64(int64_t v, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int64_t t = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += t;
    }
    return v;
}

// Total pages of the launch (every lane of the warp returns it).
__device__ int64_t total_pages(const AttnParams& p, int lane, int32_t cap) {
    int64_t tot = 0;
    for (int32_t base = 0; base < p.num_reqs; base += 32) {
        const int32_t r = base + lane;
        tot += warp_sum64(r < p.num_reqs ? req_pages(p, r, cap) : 0);
    }
    return tot;
}

// Position in the flattened (row, kv head, page) sequence.
struct Cursor {
    int64_t seg_start;  // flattened index of the segment's first page
    int32_t req, n, g, pp, kv_len, pages;  // n: first row of the group, kv_len: its last row's keys
    int32_t nr;                            // rows in the group
};

// Cursor of flattened page x (< total). Warp-collective; all lanes agree.
__device__ void locate(const AttnParams& p, int lane, int64_t x, int32_t cap, Cursor& c) {
    int64_t done = 0;
    c.req = -1;
    for (int32_t base = 0; base < p.num_reqs; base += 32) {
        const int32_t r = base + lane;
        const int64_t v = r < p.num_reqs ? req_pages(p, r, cap) : 0;
        const int64_t incl = warp_incl_scan64(v, lane);
        const int64_t chunk = __shfl_sync(0xffffffffu, incl, 31);
        if (done + chunk > x) {
            const unsigned m = __ballot_sync(0xffffffffu, done + incl > x);
            const int src = __ffs(m) - 1;
            int64_t off = done + __shfl_sync(0xffffffffu, incl - v, src);
            const int32_t req = base + src;
            const int32_t c0 = __ldg(p.cqsl + req), c1 = __ldg(p.cqsl + req + 1);
            const int32_t k = c1 - c0, seq = __ldg(p.seq_lens + req), hi = min(c1, p.max_rows);
            for (int32_t n = c0; n < hi; n += p.rg) {
                const int32_t nr = min(p.rg, hi - n);
                const int32_t kv = group_kv(seq, k, c0, n, nr);
                const int32_t pg = row_pages(kv, cap, p.block_size);
                const int64_t seg_pages = static_cast<int64_t>(pg) * p.H_kv;
                if (x < off + seg_pages) {
                    const int64_t rel = x - off;
                    c.req = req;
                    c.n = n;
                    c.nr = nr;
                    c.kv_len = min(kv, cap);
                    c.pages = pg;
                    c.g = static_cast<int32_t>(rel / pg);
                    c.pp = static_cast<int32_t>(rel - static_cast<int64_t>(c.g) * pg);
                    c.seg_start = off + static_cast<int64_t>(c.g) * pg;
                    return;
                }
                off += seg_pages;
            }
            return;
        }
        done += chunk;
    }
}

// Next page in the flattened order (skips groups without keys). RG = false:
// the launch has no row groups (p.rg == 1, every group one row).
template <bool RG = true>
__device__ __forceinline__ void advance(const AttnParams& p, Cursor& c, int32_t cap) {
    if (++c.pp < c.pages) return;
    c.seg_start += c.pages;
    c.pp = 0;
    if (++c.g < p.H_kv) return;
    c.g = 0;
    for (;;) {
        c.n += RG ? c.nr : 1;
        if (c.n >= p.max_rows) return;
        while (c.req + 1 < p.num_reqs && __ldg(p.cqsl + c.req + 1) <= c.n) ++c.req;
        const int32_t c0 = __ldg(p.cqsl + c.req), c1 = __ldg(p.cqsl + c.req + 1);
        if (c.n >= c1) return;
        // groups start at c0, c0 + rg, ...: c.n is the next one of this request
        if (RG) c.nr = min(p.rg, min(c1, p.max_rows) - c.n);
        const int32_t kv = group_kv(__ldg(p.seq_lens + c.req), c1 - c0, c0, c.n, RG ? c.nr : 1);
        c.pages = row_pages(kv, cap, p.block_size);
        c.kv_len = min(kv, cap);
        if (c.pages > 0) return;
    }
}

// Previous page in the flattened order (skips groups without keys).
template <bool RG = true>
__device__ __forceinline__ void retreat(const AttnParams& p, Cursor& c, int32_t cap) {
    if (--c.pp >= 0) return;
    if (--c.g >= 0) {  // same row, previous kv head
        c.pp = c.pages - 1;
        c.seg_start -= c.pages;
        return;
    }
    for (;;) {
        // the group ending at row c.n - 1
        const int32_t x = c.n - 1;
        if (x < 0) return;
        while (c.req > 0 && __ldg(p.cqsl + c.req) > x) --c.req;
        const int32_t c0 = __ldg(p.cqsl + c.req), c1 = __ldg(p.cqsl + c.req + 1);
        if (RG) {
            c.n = c0 + (x - c0) / p.rg * p.rg;
            c.nr = min(p.rg, min(c1, p.max_rows) - c.n);
        } else {
            c.n = x;
        }
        const int32_t kv = group_kv(__ldg(p.seq_lens + c.req), c1 - c0, c0, c.n, RG ? c.nr : 1);
        const int32_t pg = row_pages(kv, cap, p.block_size);
        if (pg > 0) {
            c.pages = pg;
            c.kv_len = min(kv, cap);
            c.g = p.H_kv - 1;
            c.pp = pg - 1;
            c.seg_start -= pg;
            return;
        }
    }
}

// Index of the worker (of `workers` equal slices of P) owning flattened page x.
__device__ __forceinline__ int32_t owner(int64_t x, int64_t P, int32_t workers) {
    return static_cast<int32_t>(((x + 1) * workers - 1) / P);
}

// Most CTAs the grid may have (it has one CTA per SM).
constexpr int kMaxCtas = 1024;

struct PieceHdr {
    int64_t s0, s1;    // segment [first page, end) in the flattened order
    const float* o;    // [virtual heads][D] partial output: in the warp's ring or in the workspace
    const float2* ml;  // [virtual heads] (m, l)
    int32_t n, g, nr;  // first row, kv head, rows of the group
    int32_t valid;
};

// ------------------------------------------------------------ per-step plan
//
// Where each warp's walk starts depends only on the step's metadata
// (cross_query_start_loc, seq_lens, block_table) and the launch shape, and
// every cross-decoder layer of a step walks the same cache with the same
// metadata. attn_tc_plan works it out once per step; each layer's launch then
// reads one 64-byte record per warp (its starting cursor and the block-table
// entries of its first pages) instead of scanning the metadata, so its first
// page copies leave after one dependent load.

constexpr int kPlanBlk = 6;  // block-table entries of a walk's first pages kept in the plan
constexpr uint32_t kPlanMagic = 0x594f434fu;

struct __align__(16) WarpPlan {
    int64_t P;          // pages of the launch
    int64_t seg_start;  // cursor of the walk's first page (see Cursor)
    int32_t req, n, g, pp, kv_len, pages;  // g: kv head | (rows of the group << 16)
    int32_t blk[kPlanBlk];  // block-table entries of the walk's first pages
};
static_assert(sizeof(WarpPlan) == 64, "one plan record is four 16-byte loads");

// The shapes a plan was made for: a launch checks them before it trusts the plan.
struct __align__(16) PlanHdr {
    uint32_t magic;
    int32_t num_reqs, max_rows, H_kv, G, block_size, max_blocks, nw, ctas, stages, d;
    int32_t rg;
    int32_t pad[4];
};
static_assert(sizeof(PlanHdr) == 64, "plan header size");

// The segments holding a CTA's first and last page, as seen by that CTA
// (read at the end of the launch by the cross-CTA merge).
struct __align__(16) CtaHdr {
    int64_t P;       // pages of the launch
    int64_t a0, a1;  // segment of the first page [first, end); a0 < 0: slice starts past the end
    int64_t b0, b1;  // segment of the last page; b0 < 0: empty slice
    int32_t an, ag;  // (first row, kv head) of segment a
    int32_t bn, bg;  // (first row, kv head) of segment b
    int32_t anr, bnr;  // rows of the groups of segments a and b
};
static_assert(sizeof(CtaHdr) == 64, "CTA header size");

// Workspace carve-up (every part a multiple of 16 bytes):
//   plan header, forward and reverse WarpPlan records [2][C][NW], CtaHdr [C],
//   arrival counters [C] (one per CTA, used by the segment starting in it),
//   partial outputs: [W][VS][D] (each warp's one mid-slice piece), then
//   [C][2][VS][D] (each CTA's first / last segment), and their (m, l) in the
//   same order, VS = p.vhs virtual heads per slot. A warp's slice-end piece
//   stays in its ring.
struct TcWs {
    PlanHdr* plan;
    WarpPlan* wplan;  // [2][C * NW]: forward walks, then reverse walks
    CtaHdr* hdr;
    uint32_t* cnt;
    float* w_o;
    float* c_o;
    float2* w_ml;
    float2* c_ml;
};

__host__ __device__ __forceinline__ int64_t tc_pieces(int64_t ctas, int nw, int VS) {
    return (ctas * nw + 2 * ctas) * VS;
}

__host__ __device__ __forceinline__ int64_t tc_plan_bytes(int64_t ctas, int nw) {
    return static_cast<int64_t>(sizeof(PlanHdr)) + 2 * ctas * nw * sizeof(WarpPlan) +
           ctas * sizeof(CtaHdr) + ((ctas * 4 + 15) & ~15ll);
}

// p.ws_o is the start of the workspace (16-byte aligned).
__device__ __forceinline__ TcWs tc_ws(const AttnParams& p, int ctas, int nw, int D) {
    TcWs w;
    uint8_t* base = reinterpret_cast<uint8_t*>(p.ws_o);
    w.plan = reinterpret_cast<PlanHdr*>(base);
    w.wplan = reinterpret_cast<WarpPlan*>(base + sizeof(PlanHdr));
    w.hdr = reinterpret_cast<CtaHdr*>(w.wplan + 2ll * ctas * nw);
    w.cnt = reinterpret_cast<uint32_t*>(w.hdr + ctas);
    float* o = reinterpret_cast<float*>(base + tc_plan_bytes(ctas, nw));
    const int64_t W = static_cast<int64_t>(ctas) * nw;
    w.w_o = o;
    w.c_o = o + W * p.vhs * D;
    w.w_ml = reinterpret_cast<float2*>(o + tc_pieces(ctas, nw, p.vhs) * D);
    w.c_ml = w.w_ml + W * p.vhs;
    return w;
}

__device__ __forceinline__ bool plan_matches(const PlanHdr& h, const AttnParams& p, int D,
                                             int BS, int nw, int stages, int ctas) {
    return h.magic == kPlanMagic && h.num_reqs == p.num_reqs && h.max_rows == p.max_rows &&
           h.H_kv == p.H_kv && h.G == p.G && h.block_size == BS && h.max_blocks == p.max_blocks &&
           h.nw == nw && h.ctas == ctas && h.stages == stages && h.d == D && h.rg == p.rg;
}

// Cursor of the first page of a walk over flattened pages [lo, hi) (forward:
// lo, reverse: hi - 1), with the block-table entries of its first pages.
// Warp-collective; lane 0 writes the record.
__device__ void plan_walk(const AttnParams& p, int lane, int64_t P, int64_t lo, int64_t hi,
                          bool rev, int32_t cap, WarpPlan* out) {
    Cursor c;
    c.req = -1;
    c.seg_start = 0;
    c.n = c.g = c.pp = c.kv_len = c.pages = 0;
    c.nr = 1;
    int32_t blk[kPlanBlk];
#pragma unroll
    for (int i = 0; i < kPlanBlk; ++i) blk[i] = -1;
    const int64_t n_my = hi - lo;
    if (n_my > 0) {
        locate(p, lane, rev ? hi - 1 : lo, cap, c);
        if (c.req >= 0) {
            Cursor w = c;
#pragma unroll
            for (int i = 0; i < kPlanBlk; ++i) {
                if (i >= n_my) break;
                blk[i] = __ldg(p.block_table + static_cast<int64_t>(w.req) * p.max_blocks + w.pp);
                if (rev) retreat(p, w, cap);
                else advance(p, w, cap);
            }
        }
    }
    if (lane == 0) {
        out->P = P;
        out->seg_start = c.seg_start;
        out->req = c.req;
        out->n = c.n;
        out->g = c.g | (c.nr << 16);  // kv head, and the rows of the group above it
        out->pp = c.pp;
        out->kv_len = c.kv_len;
        out->pages = c.pages;
#pragma unroll
        for (int i = 0; i < kPlanBlk; ++i) out->blk[i] = blk[i];
    }
}

// The per-step plan: one CTA per attention CTA, one warp per attention worker.
// Reads the metadata, then (after the dependency wait, since the previous
// kernel may be a layer still using the workspace) writes the records, the
// CTA headers and zeroes the arrival counters.
template <int NW, int STAGES, int D, int BS>
__global__ void __launch_bounds__(NW * 32) attn_tc_plan(const AttnParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const TcWs ws = tc_ws(p, gridDim.x, NW, D);
    const int64_t cap64 = static_cast<int64_t>(p.max_blocks) * BS;
    const int32_t cap = cap64 > 0x7fffffff ? 0x7fffffff : static_cast<int32_t>(cap64);
    const int64_t P = total_pages(p, lane, cap);
    const int64_t C = gridDim.x;
    const int64_t cta_lo = P * blockIdx.x / C, cta_hi = P * (blockIdx.x + 1) / C;
    const int64_t my_lo = cta_lo + (cta_hi - cta_lo) * warp / NW;
    const int64_t my_hi = cta_lo + (cta_hi - cta_lo) * (warp + 1) / NW;
    // header fields: warp 0 the segment of page cta_lo, warp 1 that of page cta_hi - 1
    int64_t hs0 = -1, hs1 = -1;
    int32_t hn = 0, hg = 0, hnr = 1;
    if (warp <= 1) {
        const int64_t x = warp == 0 ? cta_lo : cta_hi - 1;
        const bool any = warp == 0 ? cta_lo < P : cta_hi > cta_lo;
        if (any) {
            Cursor h;
            locate(p, lane, x, cap, h);
            if (h.req >= 0) {
                hs0 = h.seg_start;
                hs1 = h.seg_start + h.pages;
                hn = h.n;
                hg = h.g;
                hnr = h.nr;
            }
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t wid = static_cast<int64_t>(blockIdx.x) * NW + warp;
    plan_walk(p, lane, P, my_lo, my_hi, false, cap, ws.wplan + wid);
    plan_walk(p, lane, P, my_lo, my_hi, true, cap, ws.wplan + C * NW + wid);
    if (lane == 0 && warp <= 1) {
        CtaHdr* hp = ws.hdr + blockIdx.x;
        if (warp == 0) {
            hp->P = P;
            hp->a0 = hs0;
            hp->a1 = hs1;
            hp->an = hn;
            hp->ag = hg;
            hp->anr = hnr;
        } else {
            hp->b0 = hs0;
            hp->b1 = hs1;
            hp->bn = hn;
            hp->bg = hg;
            hp->bnr = hnr;
        }
    }
    if (threadIdx.x == 0) {
        ws.cnt[blockIdx.x] = 0u;
        if (blockIdx.x == 0) {
            PlanHdr h = {};
            h.magic = kPlanMagic;
            h.num_reqs = p.num_reqs;
            h.max_rows = p.max_rows;
            h.H_kv = p.H_kv;
            h.G = p.G;
            h.block_size = BS;
            h.max_blocks = p.max_blocks;
            h.nw = NW;
            h.ctas = static_cast<int32_t>(C);
            h.stages = STAGES;
            h.d = D;
            h.rg = p.rg;
            *ws.plan = h;
        }
    }
}

// ------------------------------------------------------- cross-CTA arrival
//
// The CTAs that share a segment cut by CTA boundaries meet at a counter kept
// by the segment's first CTA: that CTA adds 2^31 - (n - 1), the n - 1 others
// add 1, so the counter's top bit flips exactly when the last of them
// arrives, and its low 31 bits are back to zero for the next launch (the
// plan zeroes the counters once). A CTA has arrived at all of its (at most
// two) counters before it waits on any, so the waits cannot form a cycle;
// every CTA of the grid is resident (one per SM), and each wait is bounded.

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Spin until the top bit of *cnt differs from that of `old`; false on give-up.
__device__ __forceinline__ bool wait_flip(const uint32_t* cnt, uint32_t old, uint64_t limit_ns) {
    if ((ld_acquire_u32(cnt) ^ old) & 0x80000000u) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1; it < (1u << 26); ++it) {
        if ((ld_acquire_u32(cnt) ^ old) & 0x80000000u) return true;
        if ((it & 15u) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// Finishes the segments cut by CTA boundaries, inside the split kernel.
//
// Each CTA holding pages of such a segment (a holder) has written its
// CTA-level partial (m, l, o) to the workspace; it arrives at the segment's
// counter and, once every holder has arrived, takes an equal share of the
// segment's G x D outputs and combines all holders' partials for it in holder
// order (so the result depends only on logical page positions). A CTA holds
// at most two such segments (those of its first and last page); with two, the
// two halves of the CTA work on them at the same time.
//
// The share is finished with one round of global loads: every (holder,
// output) value and every (holder, head) statistic of the share is loaded at
// once into `scratch` (the CTA's ring, idle by now), then the factors and
// sums are formed in shared memory in a fixed order.
__device__ __forceinline__ uint32_t atom_add_release_u32(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.add.release.gpu.global.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(p), "r"(v)
                 : "memory");
    return old;
}

// Largest scratch (floats, a multiple of 4) one segment's share needs with H
// holders: the share's outputs of every holder (shares are whole 16-byte
// vectors: at most G*D + 4H), 3 floats per (holder, head) it touches (at most
// 2 heads once H >= G, else at most G/H + 3) and one per head.
__host__ __device__ __forceinline__ int merge_scratch_floats(int ctas, int G, int D) {
    return (G * D + 10 * ctas + 14 * (G + 1) + 4 + 3) & ~3;
}

template <int D, bool RG>
__device__ __forceinline__ void cross_cta_merge(const AttnParams& p, const TcWs& ws,
                                                const CtaHdr& Hc, float* scratch) {
    const int32_t c = blockIdx.x, ctas = gridDim.x;
    const int nthr = static_cast<int>(blockDim.x);
    const int64_t P = Hc.P;
    if (P <= 0) return;
    const int G = p.G, VS = p.vhs;  // heads of a kv group; virtual heads per partial slot
    if (!(P * c / ctas < P * (c + 1) / ctas)) return;  // a CTA without pages holds no partial

    // The (at most two) cut segments: {first page, row, kv head, first CTA,
    // holders, this CTA's rank among them}. Holders are the CTAs of the span
    // with pages: all of them when P >= ctas; otherwise each holder has
    // exactly one page of the segment and holder j owns page s0 + j.
    struct Seg {
        int64_t s0;
        int32_t n, g, nr, cf, nsh, rank;
    };
    Seg sg0 = {}, sg1 = {};
    int nseg = 0;
    const bool dense = P >= ctas;
#pragma unroll
    for (int which = 0; which < 2; ++which) {
        const int64_t s0 = which == 0 ? Hc.a0 : Hc.b0, s1 = which == 0 ? Hc.a1 : Hc.b1;
        if (s0 < 0 || (which == 1 && s0 == Hc.a0)) continue;
        const int32_t c_first = owner(s0, P, ctas), c_last = owner(s1 - 1, P, ctas);
        // not cut (finished above), or this CTA holds none of it
        if (c_first == c_last || c < c_first || c > c_last) continue;
        Seg x;
        x.s0 = s0;
        x.n = which == 0 ? Hc.an : Hc.bn;
        x.g = which == 0 ? Hc.ag : Hc.bg;
        x.nr = which == 0 ? Hc.anr : Hc.bnr;
        x.cf = c_first;
        x.nsh = dense ? c_last - c_first + 1 : static_cast<int32_t>(s1 - s0);
        x.rank = dense ? c - c_first : static_cast<int32_t>(P * c / ctas - s0);
        if (nseg == 0) sg0 = x;
        else sg1 = x;
        ++nseg;
    }
    if (nseg == 0) return;

    // arrive at every counter (release: this CTA's partials, written before
    // the barrier above, are published with it), then wait on each (acquire)
    int* ok_flag = reinterpret_cast<int*>(scratch);
    if (threadIdx.x == 0) {
        const uint32_t old0 =
            atom_add_release_u32(ws.cnt + sg0.cf, c == sg0.cf ? 0x80000000u - (sg0.nsh - 1) : 1u);
        const uint32_t old1 =
            nseg == 2 ? atom_add_release_u32(ws.cnt + sg1.cf,
                                             c == sg1.cf ? 0x80000000u - (sg1.nsh - 1) : 1u)
                      : 0u;
        bool ok = wait_flip(ws.cnt + sg0.cf, old0, kWaitLimitNs);
        if (ok && nseg == 2) ok = wait_flip(ws.cnt + sg1.cf, old1, kWaitLimitNs);
        if (!ok) set_err(p.err, YOCO_DEVERR_TIMEOUT);
        *ok_flag = ok ? 1 : 0;
    }
    __syncthreads();
    if (!*ok_flag) return;

    const int half = nseg == 2 ? nthr / 2 : nthr;  // whole warps: the warp count is even
    const int si = nseg == 2 ? static_cast<int>(threadIdx.x) / half : 0;
    const int tl = static_cast<int>(threadIdx.x) - si * half;  // thread index within the half
    const Seg sg = si == 0 ? sg0 : sg1;
    const int nh_ = sg.nsh;
    // this CTA's share of the segment's (rows x G) x D outputs (whole 16-byte
    // vectors), and the virtual heads (row-major over the group's rows) it touches
    const int total = (RG ? sg.nr : 1) * G * D;
    const int per = ((total + nh_ - 1) / nh_ + 3) & ~3;
    const int lo = min(total, sg.rank * per), hi = min(total, lo + per);
    const int nout = hi - lo, nv = nout >> 2;
    const int h_lo = lo / D, nhd = nout > 0 ? (hi - 1) / D - h_lo + 1 : 0;
    float* so = scratch + 16 + si * merge_scratch_floats(ctas, VS, D);  // [holder][nout]
    float2* sml = reinterpret_cast<float2*>(so + nh_ * nout);          // [holder][nhd]
    float* sf = reinterpret_cast<float*>(sml + nh_ * nhd);             // [holder][nhd] 2^(m - M)
    float* sInvL = sf + nh_ * nhd;                                     // [nhd]
    // holder j's partial slot: the segment begins in holder 0's slice (slot 1);
    // for every other holder it is the first segment (slot 0)
    auto slot = [&](int j) -> int64_t {
        const int64_t cj = dense ? sg.cf + j : owner(sg.s0 + j, P, ctas);
        return (cj * 2 + (j == 0 ? 1 : 0)) * VS;
    };
    // One round of asynchronous global -> shared copies: every holder's
    // outputs of the share (16-byte vectors) and (m, l) of its heads. The
    // loops stay rolled: this code runs once per launch, where instruction
    // fetch, not the copies, sets the time.
#pragma unroll 1
    for (int j = tl; j < nh_ * nv; j += half) {
        const int hj = j / nv, v = j - hj * nv;
        cp_async_16(so + hj * nout + 4 * v, ws.c_o + slot(hj) * D + lo + 4 * v);
    }
#pragma unroll 1
    for (int k = tl; k < nh_ * nhd; k += half) {
        const int hj = k / nhd;
        cp_async_8(sml + k, ws.c_ml + slot(hj) + h_lo + (k - hj * nhd));
    }
    cp_async_wait_all();
    __syncthreads();
    // factors: for each head of the share, M = max over holders, f_j = 2^(m_j - M),
    // L = sum l_j f_j. One warp per head, lanes over holders; the reductions
    // are fixed butterfly trees, so the result does not depend on timing.
    const int nwh = half >> 5, wl = tl >> 5, ln = tl & 31;
#pragma unroll 1
    for (int hh = wl; hh < nhd; hh += nwh) {
        float M = -INFINITY;
#pragma unroll 1
        for (int j = ln; j < nh_; j += 32) M = fmaxf(M, sml[j * nhd + hh].x);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float L = 0.f;
#pragma unroll 1
        for (int j = ln; j < nh_; j += 32) {
            const float2 ml = sml[j * nhd + hh];
            const float f = ml.x != -INFINITY ? exp2_approx(ml.x - M) : 0.f;
            sf[j * nhd + hh] = f;
            L += ml.y * f;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
        if (ln == 0) sInvL[hh] = 1.f / L;
    }
    __syncthreads();
    __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(p.out);
    // a holder with no key has f = 0 and a slot never written: select, not 0 * x
    auto term = [&](int j, int e, int hh) {
        const float f = sf[j * nhd + hh];
        return f != 0.f ? so[j * nout + e] * f : 0.f;
    };
#pragma unroll 1
    for (int e = tl; e < nout; e += half) {
        const int hh = (lo + e) / D - h_lo;
        // four independent chains over the holders (j mod 4), summed in a fixed order
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        int j = 0;
#pragma unroll 1
        for (; j + 4 <= nh_; j += 4) {
            a0 += term(j, e, hh);
            a1 += term(j + 1, e, hh);
            a2 += term(j + 2, e, hh);
            a3 += term(j + 3, e, hh);
        }
#pragma unroll 1
        for (; j < nh_; ++j) a0 += term(j, e, hh);
        int64_t dst = (static_cast<int64_t>(sg.n) * p.H_q + sg.g * G) * D + lo + e;
        if constexpr (RG) {
            if (!(sInvL[hh] < INFINITY)) continue;  // a group row without keys: zero-filled in the kernel
            // virtual head v = (row of the group) * G + head
            const int v = (lo + e) / D, d = lo + e - v * D;
            dst = ((static_cast<int64_t>(sg.n) + v / G) * p.H_q + sg.g * G + v % G) * D + d;
        }
        outp[dst] = __float2bfloat16_rn(((a0 + a1) + (a2 + a3)) * sInvL[hh]);
    }
}

// --------------------------------------------------------------- kernel

// FUSE: fused decode step (append this step's tokens, patch them into the
// copied pages); instantiated with REV = false only.
// RG: cross rows grouped on one walk (p.rg > 1; FUSE = false only).
// Without it every segment is one row and the per-column causal masks and
// the guard for columns without keys compile away.
// PR: warp pairs (NT = 1, FUSE = false): a worker is two warps that walk one
// slice from one ring, warp 2k taking columns 0-7 of the group and warp
// 2k + 1 columns 8-15. The pair's leader issues the copies; both wait on them
// and agree on every outcome through one pair barrier, so that they always
// take the same path.
template <int D, int BS, int NT, bool REV, bool F8, bool FUSE, bool RG, bool PR>
__global__ void __launch_bounds__(TcShape<D, BS, F8, NT, PR>::NW * 32, 1)
    attn_tc_persistent(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
    using S = TcShape<D, BS, F8, NT, PR>;
    constexpr int NW = S::NW, WK = S::WK, STAGES = S::STAGES, NTG = S::NTG;
    static_assert(S::PIECE_PAIR <= STAGES * S::STAGE_BYTES,
                  "a worker's two end-of-slice pieces must fit in its ring");
    static_assert(!F8 || D % 128 == 0, "e4m3 pages need 128-byte rows");
    static_assert(!RG || !FUSE, "the fused decode step has one row per request");
    static_assert(!PR || !FUSE, "the fused decode step runs one warp per ring");
    // the cross-CTA merge splits the CTA into two halves for its two segments,
    // each made of whole warps (its warp shuffles take full masks)
    static_assert(NW % 2 == 0, "an even number of warps per CTA");
    static_assert(WK <= 15, "one named barrier per pair");
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[WK * STAGES];
    __shared__ int32_t stage_blk[WK * STAGES];  // physical page of each stage (-1: invalid)
    // e4m3: the page's scale record {k_scale, v_scale, -, -}, copied with the page
    __shared__ __align__(16) float4 stage_scale[F8 ? WK * STAGES : 1];
    __shared__ PieceHdr hdr[WK][2];
    __shared__ int abort_flag;
    __shared__ __align__(16) CtaHdr cta_hdr;  // this CTA's first / last segment (from the plan)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gl = lane >> 2, tq = lane & 3;  // mma fragment row group / column pair
    const int wk = PR ? warp >> 1 : warp;    // this warp's worker
    const int c8 = PR ? (warp & 1) * 8 : 0;  // first column of the group this warp takes
    const bool leader = !PR || (warp & 1) == 0;
    const int pair_bar = 1 + wk;             // the pair's named barrier (PR)
    const TcWs ws = tc_ws(p, gridDim.x, WK, D);
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* wbuf = smem + wk * STAGES * S::STAGE_BYTES;
    uint64_t* wbar = bars + wk * STAGES;
    if (lane == 0 && leader) {  // each worker's ring barriers: only its warps wait on them
        for (int i = 0; i < STAGES; ++i) mbar_init(&wbar[i], 1);
        fence_mbar_init();
        hdr[wk][0].valid = hdr[wk][1].valid = 0;
    }
    __syncwarp();
    // This warp's plan record (the forward or the reverse walk): four
    // independent loads, the only dependent step before the first page copies.
    static_assert(STAGES <= kPlanBlk, "the plan holds the block ids of the prologue's pages");
    uint4 r0, r1, r2, r3;
    {
        const uint4* src = reinterpret_cast<const uint4*>(
            ws.wplan + (REV ? static_cast<int64_t>(gridDim.x) * WK : 0) +
            static_cast<int64_t>(blockIdx.x) * WK + wk);
        r0 = __ldg(src);
        r1 = __ldg(src + 1);
        r2 = __ldg(src + 2);
        r3 = __ldg(src + 3);
    }
    int plan_state = 0;  // thread 0: 0 plan usable, 1 launch already aborted, 2 no matching plan
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        const uint4* hs = reinterpret_cast<const uint4*>(ws.plan);
        const uint4* cs = reinterpret_cast<const uint4*>(ws.hdr + blockIdx.x);
        uint4 h[4], c[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            h[i] = __ldg(hs + i);
            c[i] = __ldg(cs + i);
        }
        PlanHdr ph;
        ph.magic = h[0].x;
        ph.num_reqs = static_cast<int32_t>(h[0].y);
        ph.max_rows = static_cast<int32_t>(h[0].z);
        ph.H_kv = static_cast<int32_t>(h[0].w);
        ph.G = static_cast<int32_t>(h[1].x);
        ph.block_size = static_cast<int32_t>(h[1].y);
        ph.max_blocks = static_cast<int32_t>(h[1].z);
        ph.nw = static_cast<int32_t>(h[1].w);
        ph.ctas = static_cast<int32_t>(h[2].x);
        ph.stages = static_cast<int32_t>(h[2].y);
        ph.d = static_cast<int32_t>(h[2].z);
        ph.rg = static_cast<int32_t>(h[2].w);
        uint4* cd = reinterpret_cast<uint4*>(&cta_hdr);
#pragma unroll
        for (int i = 0; i < 4; ++i) cd[i] = c[i];
        plan_state = launch_aborted(p) ? 1
                     : plan_matches(ph, p, D, BS, WK, STAGES, static_cast<int>(gridDim.x)) ? 0 : 2;
    }
    const int64_t P = static_cast<int64_t>((static_cast<uint64_t>(r0.y) << 32) | r0.x);
    const int64_t C = gridDim.x;
    const int64_t cta_lo = P * blockIdx.x / C, cta_hi = P * (blockIdx.x + 1) / C;
    const int64_t my_lo = cta_lo + (cta_hi - cta_lo) * wk / WK;
    const int64_t my_hi = cta_lo + (cta_hi - cta_lo) * (wk + 1) / WK;
    int32_t n_my = static_cast<int32_t>(my_hi - my_lo);
    const int32_t wid = blockIdx.x * WK + wk;
    const int64_t cap64 = static_cast<int64_t>(p.max_blocks) * BS;
    const int32_t cap = cap64 > 0x7fffffff ? 0x7fffffff : static_cast<int32_t>(cap64);

    // Odd layers may walk each slice backwards (REV): a layer then starts on
    // the pages the previous layer read last, which are still in L2.
    constexpr bool rev = REV;
    auto step = [&](Cursor& c) {
        if (rev) retreat<RG>(p, c, cap);
        else advance<RG>(p, c, cap);
    };
    Cursor cc;  // page being consumed
    cc.seg_start = static_cast<int64_t>((static_cast<uint64_t>(r0.w) << 32) | r0.z);
    cc.req = static_cast<int32_t>(r1.x);
    cc.n = static_cast<int32_t>(r1.y);
    cc.g = static_cast<int32_t>(r1.z & 0xffffu);
    cc.nr = RG ? static_cast<int32_t>(r1.z >> 16) : 1;
    cc.pp = static_cast<int32_t>(r1.w);
    cc.kv_len = static_cast<int32_t>(r2.x);
    cc.pages = static_cast<int32_t>(r2.y);
    const int32_t plan_blk[kPlanBlk] = {static_cast<int32_t>(r2.z), static_cast<int32_t>(r2.w),
                                        static_cast<int32_t>(r3.x), static_cast<int32_t>(r3.y),
                                        static_cast<int32_t>(r3.z), static_cast<int32_t>(r3.w)};
    // A record that does not describe a page of this launch (a plan for other
    // metadata, or none) must not steer a copy: nothing is issued, and the
    // header check below ends the launch.
    const bool rec_ok = P >= 0 && cc.req >= 0 && cc.req < p.num_reqs && cc.g >= 0 &&
                        cc.g < p.H_kv && cc.nr >= 1 && cc.nr <= p.rg && cc.n >= 0 &&
                        cc.n + cc.nr <= p.max_rows && cc.pages > 0 &&
                        cc.pp >= 0 && cc.pp < cc.pages && static_cast<int64_t>(cc.pages) * BS <= cap64 + BS;
    if (!rec_ok || n_my < 0) n_my = 0;
    Cursor pc = cc;  // next page to issue (lane 0)
    // lane 0: block-table entry of page pc, loaded one issue ahead so that its
    // latency overlaps the page computed in between
    int32_t blk_next = -1;
    auto fetch_blk = [&]() {
        blk_next = __ldg(p.block_table + static_cast<int64_t>(pc.req) * p.max_blocks + pc.pp);
    };

    // With keep_tail, the pages are streamed through L2 with an evict-first
    // hint except the last keep_pages of this warp's walk (evict-last): about
    // kKeepBytes over the grid stay in L2 for the next layer, which walks the
    // other way and starts on them.
    constexpr int64_t kKeepBytes = (F8 ? 20ll : 40ll) << 20;
    const bool keep_tail = p.keep_tail != 0;
    const uint64_t pol_keep = keep_tail ? make_l2_policy_evict_last() : 0;
    const uint64_t pol_stream = keep_tail ? make_l2_policy_evict_first() : 0;
    const int keep_pages = static_cast<int>(
        kKeepBytes / (static_cast<int64_t>(gridDim.x) * WK * S::STAGE_BYTES));
    auto issue = [&](int i) {  // the worker's lane 0 only; pc is at page i, blk_next its entry
        const int st = i % STAGES;
        uint64_t* bar = wbar + st;
        const int32_t blk = blk_next;
        // published to the consumer lanes by the barrier's release/acquire
        stage_blk[wk * STAGES + st] = (blk < 0 || blk >= p.num_blocks) ? -1 : blk;
        if (blk < 0 || blk >= p.num_blocks) {
            set_err(p.err, YOCO_DEVERR_PAGE_RANGE);
            mbar_arrive(bar);
        } else {
            mbar_arrive_expect_tx(bar, 2 * S::PAGE_BYTES + (F8 ? 16 : 0));
            uint8_t* kd = wbuf + st * S::STAGE_BYTES;
            uint8_t* vd = kd + S::PAGE_BYTES;
            const int32_t y = (blk * p.H_kv + pc.g) * BS;
            if (keep_tail) {
                const uint64_t pol = i >= n_my - keep_pages ? pol_keep : pol_stream;
#pragma unroll
                for (int c = 0; c < S::KSUB; ++c) {
                    tma_load_2d_hint(kd + c * S::SUB_BYTES, &tm_k, c * S::SUBE, y, bar, pol);
                    tma_load_2d_hint(vd + c * S::SUB_BYTES, &tm_v, c * S::SUBE, y, bar, pol);
                }
            } else {
#pragma unroll
                for (int c = 0; c < S::KSUB; ++c) {
                    tma_load_2d(kd + c * S::SUB_BYTES, &tm_k, c * S::SUBE, y, bar);
                    tma_load_2d(vd + c * S::SUB_BYTES, &tm_v, c * S::SUBE, y, bar);
                }
            }
            if constexpr (F8)
                bulk_load(&stage_scale[wk * STAGES + st],
                          p.scales + static_cast<int64_t>(blk) * p.H_kv + pc.g, 16, bar);
        }
        step(pc);
    };
    const int pro = n_my < STAGES ? n_my : STAGES;
    if (lane == 0 && leader) {
        // the prologue's pages take their block ids from the plan
#pragma unroll
        for (int i = 0; i < STAGES; ++i) {
            if (i < pro) {
                blk_next = plan_blk[i];
                issue(i);
            }
        }
        if (pro < n_my) fetch_blk();
    }
    if (threadIdx.x == 0) abort_flag = plan_state;
    __syncthreads();  // every ring's barriers initialised; the plan checked
    if (abort_flag) {
        // a launch that has already failed, or a workspace without a plan for
        // these shapes: drain the copies issued above, flag, and end
        for (int i = 0; i < pro; ++i) (void)mbar_wait_bounded(wbar + i, 0, kWaitLimitNs);
        if (threadIdx.x == 0 && abort_flag == 2) set_err(p.err, YOCO_DEVERR_PLAN);
        return;
    }
    // When launched as a programmatic dependent of the previous kernel in the
    // stream (the caller allows it only when that kernel writes neither), the
    // code above reads the metadata and the cache while that kernel drains.
    // Queries, outputs and the workspace are touched after this wait.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (FUSE && warp == NW - 1) {
        // fused decode step: append each request's one new token (requests spread
        // over the CTAs; after the wait, so no earlier kernel still reads the pools)
        constexpr int CH = F8 ? D / 16 : D / 8;  // 16-byte chunks of a cached row
        for (int32_t r = blockIdx.x; r < p.num_reqs; r += gridDim.x) {
            const int32_t q0 = __ldg(p.cqsl + r), q1 = __ldg(p.cqsl + r + 1);
            if (q1 - q0 != 1) {
                if (lane == 0) set_err(p.err, YOCO_DEVERR_OFFSETS);
                continue;
            }
            const int32_t pos = __ldg(p.seq_lens + r) - 1;
            if (pos < 0 || pos / BS >= p.max_blocks) {
                if (lane == 0) set_err(p.err, YOCO_DEVERR_POS_RANGE);
                continue;
            }
            const int32_t blk = __ldg(p.block_table + static_cast<int64_t>(r) * p.max_blocks + pos / BS);
            if (blk < 0 || blk >= p.num_blocks) {
                if (lane == 0) set_err(p.err, YOCO_DEVERR_PAGE_RANGE);
                continue;
            }
            for (int32_t h = 0; h < p.H_kv; ++h) {
                const int64_t row = (static_cast<int64_t>(blk) * p.H_kv + h) * BS + pos % BS;
                const uint4* ks = static_cast<const uint4*>(p.k_new) + (static_cast<int64_t>(q0) * p.H_kv + h) * (D / 8);
                const uint4* vs = static_cast<const uint4*>(p.v_new) + (static_cast<int64_t>(q0) * p.H_kv + h) * (D / 8);
                uint4* kd = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.k_pool) + row * D * S::ESZ);
                uint4* vd = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.v_pool) + row * D * S::ESZ);
                if constexpr (F8) {
                    const float4 sc = __ldg(p.scales + static_cast<int64_t>(blk) * p.H_kv + h);
                    if (!scale_usable(sc.x) || !scale_usable(sc.y)) {
                        if (lane == 0) set_err(p.err, YOCO_DEVERR_SCALE);
                        continue;
                    }
                    if (lane < CH) {
                        const uint2 k0 = quantise8_e4m3(__ldg(ks + 2 * lane), sc.x);
                        const uint2 k1 = quantise8_e4m3(__ldg(ks + 2 * lane + 1), sc.x);
                        const uint2 v0 = quantise8_e4m3(__ldg(vs + 2 * lane), sc.y);
                        const uint2 v1 = quantise8_e4m3(__ldg(vs + 2 * lane + 1), sc.y);
                        kd[lane] = make_uint4(k0.x, k0.y, k1.x, k1.y);
                        vd[lane] = make_uint4(v0.x, v0.y, v1.x, v1.y);
                    }
                } else if (lane < CH) {
                    kd[lane] = __ldg(ks + lane);
                    vd[lane] = __ldg(vs + lane);
                }
            }
        }
    }
    if (warp == NW - 1) {
        // rows with no key to attend: zero output, flag (requests spread over the CTAs)
        __nv_bfloat16* const outz = static_cast<__nv_bfloat16*>(p.out);
        for (int32_t r = blockIdx.x; r < p.num_reqs; r += gridDim.x) {
            const int32_t c0 = __ldg(p.cqsl + r), c1 = __ldg(p.cqsl + r + 1);
            const int32_t seq = __ldg(p.seq_lens + r), k = c1 - c0;
            for (int32_t n = c0; n < c1 && n < p.max_rows; ++n) {
                const int32_t kv = seq - k + (n - c0) + 1;
                if (kv <= 0) {
                    for (int i = lane; i < p.H_q * D; i += 32)
                        outz[static_cast<int64_t>(n) * p.H_q * D + i] = __float2bfloat16_rn(0.f);
                    if (lane == 0) set_err(p.err, YOCO_DEVERR_EMPTY_ROW);
                } else if ((kv > cap || kv > p.max_seq_len) && lane == 0) {
                    set_err(p.err, YOCO_DEVERR_POS_RANGE);
                }
            }
        }
    }
    uint32_t qf[S::QSM ? 1 : S::KD][NT][2];  // queries in registers (not with QSM)
    float o[S::KD][NT][4];
    float m_run[NT][2], l_part[NT][2];
    // e4m3: o holds sum p * (v_scale / vref) * code; vref is the V scale of the
    // segment's first page here, moved (and o rescaled) when a page's ratio
    // leaves [1/16, 16], so that the f16 weights stay in range
    float vref = 0.f, vinv = 0.f;
    auto reset_state = [&]() {
        vref = 0.f;
#pragma unroll
        for (int a = 0; a < S::KD; ++a)
#pragma unroll
            for (int b = 0; b < NT; ++b)
#pragma unroll
                for (int c = 0; c < 4; ++c) o[a][b][c] = 0.f;
#pragma unroll
        for (int b = 0; b < NT; ++b) {
            m_run[b][0] = m_run[b][1] = -INFINITY;
            l_part[b][0] = l_part[b][1] = 0.f;
        }
    };
    // B operand of S^T = K Q^T: head gl of n-tile nt, head dims 2tq.. of each 16-wide step.
    // e4m3 keys arrive with each lane's four consecutive head dims 4tq..4tq+3 of a
    // 16-wide step standing for k indices {2tq, 2tq+1, 2tq+8, 2tq+9}: the query takes
    // the same order (a dot product does not depend on the order of its terms),
    // rounded to f16 to match the f16 keys.
    // Virtual head v = nt * 8 + gl of a group of nr rows is head v % G of row
    // n + v / G (rows of one request share the walk; zero past nr * G).
    // moff[nt][e]: how many keys fewer than the group's last row the row of
    // accumulator column nt * 8 + 2 tq + e sees (0 past the group's rows)
    int32_t moff[NT][2];
    // QSM: the segment's queries as 16 rows (virtual heads) of D 16-bit values
    // in this warp's own shared-memory tile, 16-byte chunk j of row h at
    // h * 2D + ((j ^ (h & 7)) << 4) so that the 8 rows an ldmatrix reads fall
    // in distinct banks. For e4m3 keys each 16-dim step holds the f16 query in
    // the keys' order: chunk 2kk dims {0,1,4,5,8,9,12,13}, chunk 2kk + 1 dims
    // {2,3,6,7,10,11,14,15} (of step kk), so that a lane's ldmatrix pairs are
    // the dims its key registers hold.
    uint8_t* const qsm = smem + S::RING_BYTES + warp * S::Q_BYTES;
    auto load_q_smem = [&](int32_t n, int32_t g, int32_t nr) {
        const int nvh = RG ? nr * p.G : p.G;
        auto qsrc = [&](int h) {
            const int hr = RG ? h / p.G : 0, hh = h - hr * p.G;
            return static_cast<const __nv_bfloat16*>(p.q) +
                   ((static_cast<int64_t>(n) + hr) * p.H_q + g * p.G + hh) * D;
        };
        __syncwarp();  // the previous segment's ldmatrix reads are done
        if constexpr (F8) {
            constexpr int NB = D / 16;  // 16-dim steps per row
            static_assert(32 % NB == 0, "whole rows per pass");
#pragma unroll 1
            for (int x = lane; x < 16 * NB; x += 32) {
                const int h = x / NB, kk = x - h * NB;
                uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;
                if (h < nvh) {
                    const uint4* src = reinterpret_cast<const uint4*>(qsrc(h) + kk * 16);
                    a = __ldg(src);
                    b = __ldg(src + 1);
                }
                auto w = [](uint32_t v) { return pack_f16x2(bf16lo_to_f32(v), bf16hi_to_f32(v)); };
                uint8_t* row = qsm + h * (2 * D);
                *reinterpret_cast<uint4*>(row + (((2 * kk) ^ (h & 7)) << 4)) =
                    make_uint4(w(a.x), w(a.z), w(b.x), w(b.z));
                *reinterpret_cast<uint4*>(row + (((2 * kk + 1) ^ (h & 7)) << 4)) =
                    make_uint4(w(a.y), w(a.w), w(b.y), w(b.w));
            }
        } else {
            constexpr int NCH = D / 8;  // 16-byte chunks per row
            static_assert(32 % NCH == 0 || NCH % 32 == 0, "whole rows per pass");
#pragma unroll 1
            for (int x = lane; x < 16 * NCH; x += 32) {
                const int h = x / NCH, j = x - h * NCH;
                const uint4 v = h < nvh ? __ldg(reinterpret_cast<const uint4*>(qsrc(h)) + j)
                                        : make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(qsm + h * (2 * D) + ((j ^ (h & 7)) << 4)) = v;
            }
        }
        __syncwarp();
    };
    // this lane's ldmatrix row of the query tile: matrices (rows 0-7 | 8-15) x
    // (chunk 2kk | 2kk + 1), so the four registers are n-tile 0's b0, b1, then
    // n-tile 1's
    const uint32_t q_lane = smem_u32(qsm) + (((lane >> 4) * 8 + (lane & 7)) * (2 * D));
    auto q_addr = [&](int kk) {
        return q_lane + ((((2 * kk) + ((lane >> 3) & 1)) ^ (lane & 7)) << 4);
    };
    auto load_q = [&](int32_t n, int32_t g, int32_t nr) {
        if constexpr (S::QSM) {
            if constexpr (RG) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        moff[nt][e] = nr - 1 - min((nt * 8 + 2 * tq + e) / p.G, nr - 1);
            }
            load_q_smem(n, g, nr);
        } else {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int h = c8 + nt * 8 + gl;
                bool ok;
                int hr = 0, hh = 0;
                if constexpr (RG) {
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        moff[nt][e] = nr - 1 - min((c8 + nt * 8 + 2 * tq + e) / p.G, nr - 1);
                    ok = h < nr * p.G;
                    hr = ok ? h / p.G : 0;
                    hh = ok ? h - hr * p.G : 0;
                } else {
                    moff[nt][0] = moff[nt][1] = 0;
                    ok = h < p.G;
                    hh = ok ? h : 0;
                }
                const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(p.q) +
                                            ((static_cast<int64_t>(n) + hr) * p.H_q + g * p.G + hh) * D;
                if constexpr (F8) {
                    const uint2* src = reinterpret_cast<const uint2*>(qrow);
#pragma unroll
                    for (int kk = 0; kk < S::KD; ++kk) {
                        const uint2 v = ok ? __ldg(src + kk * 4 + tq) : make_uint2(0u, 0u);
                        qf[kk][nt][0] = pack_f16x2(bf16lo_to_f32(v.x), bf16hi_to_f32(v.x));
                        qf[kk][nt][1] = pack_f16x2(bf16lo_to_f32(v.y), bf16hi_to_f32(v.y));
                    }
                } else {
                    const uint32_t* src = reinterpret_cast<const uint32_t*>(qrow);
#pragma unroll
                    for (int kk = 0; kk < S::KD; ++kk) {
                        qf[kk][nt][0] = ok ? __ldg(src + kk * 8 + tq) : 0u;
                        qf[kk][nt][1] = ok ? __ldg(src + kk * 8 + 4 + tq) : 0u;
                    }
                }
            }
        }
    };
    reset_state();
    // Fused decode step: this lane's 16-byte chunk(s) of the segment's new token
    // row (the request's one new token), K and V, loaded when the segment starts.
    constexpr int PCH = F8 ? D / 16 : D / 8;  // 16-byte chunks of one cached token row
    constexpr int PIN = F8 ? 2 : 1;           // bf16 input words per chunk
    uint4 pk[PIN], pv[PIN];
    constexpr bool fused = FUSE;
    auto load_patch = [&](int32_t req, int32_t g) {
        const int64_t tok = __ldg(p.cqsl + req + 1) - 1;
        const uint4* kr = static_cast<const uint4*>(p.k_new) + (tok * p.H_kv + g) * (D / 8);
        const uint4* vr_ = static_cast<const uint4*>(p.v_new) + (tok * p.H_kv + g) * (D / 8);
        if (lane < PCH) {
#pragma unroll
            for (int u = 0; u < PIN; ++u) {
                pk[u] = __ldg(kr + lane * PIN + u);
                pv[u] = __ldg(vr_ + lane * PIN + u);
            }
        }
    };
    // head dim of accumulator row gl (half 0) / gl + 8 (half 1) of 16-wide step md
    auto drow = [&](int md, int half) {
        return F8 ? md * 16 + 2 * gl + half : md * 16 + gl + 8 * half;
    };
    const float sl2 = p.scale_log2;
    bool aborted = false;
    int consumed = 0;
    // one piece: [G][D] o, then [G] (m, l); 16-byte stride keeps float4 access aligned
    const int piece_bytes = (p.vhs * (D * 4 + 8) + 15) & ~15;

    for (int i = 0; i < n_my; ++i) {
        if (i == 0 || cc.pp == (rev ? cc.pages - 1 : 0)) {
            load_q(cc.n, cc.g, cc.nr);
            if (fused) load_patch(cc.req, cc.g);
        }
        const int st = i % STAGES;
        bool landed = mbar_wait_bounded(wbar + st, (i / STAGES) & 1, kWaitLimitNs);
        if constexpr (PR) landed = pair_all(pair_bar, landed);  // both warps or neither
        if (!landed) {
            aborted = true;
            break;
        }
        consumed = i + 1;
        if (stage_blk[wk * STAGES + st] >= 0) {
            const uint32_t kbase = smem_u32(wbuf + st * S::STAGE_BYTES);
            const uint32_t vbase = kbase + S::PAGE_BYTES;
            const int32_t nvalid = min(BS, cc.kv_len - cc.pp * BS);
            float sl2p = sl2, vr = 1.f;  // score factor, weight factor of this page
            if constexpr (F8) {
                // codes widen exactly; the page's K scale goes into the score factor
                const float4 sc4 = stage_scale[wk * STAGES + st];
                if (lane == 0 && !(sc4.x >= 0x1p-16f && sc4.x <= 128.f && sc4.y >= 0x1p-16f &&
                                   sc4.y <= 128.f))
                    set_err(p.err, YOCO_DEVERR_SCALE);
                sl2p = sl2 * sc4.x;
                if (vref == 0.f) {
                    vref = sc4.y;
                    vinv = 1.f / sc4.y;
                }
                vr = sc4.y * vinv;
                if (!(vr <= 16.f && vr >= 0.0625f)) {  // warp-uniform, rare
                    const float f = vref / sc4.y;
#pragma unroll
                    for (int md = 0; md < S::KD; ++md)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int c = 0; c < 4; ++c) o[md][nt][c] *= f;
                    vref = sc4.y;
                    vinv = 1.f / sc4.y;
                    vr = 1.f;
                }
            }
            if (fused && cc.pp == (cc.kv_len - 1) / BS) {
                // Fused decode step: the row's newest key is this step's token, which
                // this launch also appends to the pools; whatever the page copy
                // brought for that slot, take it from the input (quantised by the
                // append's rule for e4m3).
                const int s = (cc.kv_len - 1) % BS;
                uint8_t* kd = wbuf + st * S::STAGE_BYTES;
                if (lane < PCH) {
                    uint4 kw, vw;
                    if constexpr (F8) {
                        const float4 sc4 = stage_scale[wk * STAGES + st];
                        const uint2 k0 = quantise8_e4m3(pk[0], sc4.x), k1 = quantise8_e4m3(pk[PIN - 1], sc4.x);
                        const uint2 v0 = quantise8_e4m3(pv[0], sc4.y), v1 = quantise8_e4m3(pv[PIN - 1], sc4.y);
                        kw = make_uint4(k0.x, k0.y, k1.x, k1.y);
                        vw = make_uint4(v0.x, v0.y, v1.x, v1.y);
                    } else {
                        kw = pk[0];
                        vw = pv[0];
                    }
                    const uint32_t off = swz<BS>(lane >> 3, s, lane & 7);
                    *reinterpret_cast<uint4*>(kd + off) = kw;
                    *reinterpret_cast<uint4*>(kd + S::PAGE_BYTES + off) = vw;
                }
                fence_proxy_async_smem();  // before a later copy refills the stage
                __syncwarp();
            }
            if (nvalid < BS) {
                // Rows past the causal end may hold stale data (even NaN), and a
                // zero probability times NaN is NaN: clear those V rows first.
                // (a pair's warps clear alternate sub-tiles, then meet)
                uint8_t* vd = wbuf + st * S::STAGE_BYTES + S::PAGE_BYTES;
                const int nbytes = (BS - nvalid) * 128;
                for (int c = PR ? (warp & 1) : 0; c < S::KSUB; c += PR ? 2 : 1)
                    for (int b = lane * 16; b < nbytes; b += 32 * 16)
                        *reinterpret_cast<uint4*>(vd + c * S::SUB_BYTES + nvalid * 128 + b) =
                            make_uint4(0, 0, 0, 0);
                fence_proxy_async_smem();
                if constexpr (PR) pair_sync(pair_bar);
                else __syncwarp();
            }
            // ---- S^T = K Q^T (tokens x heads); two accumulators halve the chain ----
            float sc[S::MT][NT][4];
            {
                float sc2[S::MT][NT][4];
#pragma unroll
                for (int mt = 0; mt < S::MT; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int c = 0; c < 4; ++c) sc[mt][nt][c] = sc2[mt][nt][c] = 0.f;
                const int mi = lane >> 3, rr = lane & 7;
                if constexpr (S::QSM && F8) {
                    // as below, with the query fragments read from the warp's tile
                    // once per pair of k steps for all token tiles
#pragma unroll
                    for (int kp = 0; kp < S::KD / 2; ++kp) {
                        uint32_t qa[4], qb[4];
                        ldsm_x4(q_addr(2 * kp), qa[0], qa[1], qa[2], qa[3]);
                        ldsm_x4(q_addr(2 * kp + 1), qb[0], qb[1], qb[2], qb[3]);
#pragma unroll
                        for (int mt = 0; mt < S::MT; ++mt) {
                            const int t = mt * 16 + (mi & 1) * 8 + rr;
                            const int ch = 2 * kp + (mi >> 1);
                            uint32_t r0, r1, r2, r3;
                            ldsm_x4(kbase + swz<BS>(ch >> 3, t, ch & 7), r0, r1, r2, r3);
                            const uint32_t a0 = e4m3x2_lo_to_f16x2(r0);
                            const uint32_t a1 = e4m3x2_lo_to_f16x2(r1);
                            const uint32_t a2 = e4m3x2_hi_to_f16x2(r0);
                            const uint32_t a3 = e4m3x2_hi_to_f16x2(r1);
                            const uint32_t b0 = e4m3x2_lo_to_f16x2(r2);
                            const uint32_t b1 = e4m3x2_lo_to_f16x2(r3);
                            const uint32_t b2 = e4m3x2_hi_to_f16x2(r2);
                            const uint32_t b3 = e4m3x2_hi_to_f16x2(r3);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                mma_f16_16816(sc[mt][nt], a0, a1, a2, a3, qa[2 * nt], qa[2 * nt + 1]);
                                mma_f16_16816(sc2[mt][nt], b0, b1, b2, b3, qb[2 * nt], qb[2 * nt + 1]);
                            }
                        }
                    }
                } else if constexpr (S::QSM) {
#pragma unroll
                    for (int kk = 0; kk < S::KD; ++kk) {
                        uint32_t qk[4];
                        ldsm_x4(q_addr(kk), qk[0], qk[1], qk[2], qk[3]);
#pragma unroll
                        for (int mt = 0; mt < S::MT; ++mt) {
                            const int t = mt * 16 + (mi & 1) * 8 + rr;
                            uint32_t a0, a1, a2, a3;
                            ldsm_x4(kbase + swz<BS>(kk >> 2, t, (kk & 3) * 2 + (mi >> 1)), a0, a1,
                                    a2, a3);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                if (kk & 1)
                                    mma_bf16_16816(sc2[mt][nt], a0, a1, a2, a3, qk[2 * nt],
                                                   qk[2 * nt + 1]);
                                else
                                    mma_bf16_16816(sc[mt][nt], a0, a1, a2, a3, qk[2 * nt],
                                                   qk[2 * nt + 1]);
                            }
                        }
                    }
                } else if constexpr (F8) {
                    // one ldmatrix.x4 = 16 tokens x 32 head dims (two k steps); a lane's
                    // 32-bit register holds 4 consecutive e4m3 of one token
#pragma unroll
                    for (int mt = 0; mt < S::MT; ++mt) {
                        const int t = mt * 16 + (mi & 1) * 8 + rr;
#pragma unroll
                        for (int kp = 0; kp < S::KD / 2; ++kp) {
                            const int ch = 2 * kp + (mi >> 1);  // 16-byte chunk along head_dim
                            uint32_t r0, r1, r2, r3;
                            ldsm_x4(kbase + swz<BS>(ch >> 3, t, ch & 7), r0, r1, r2, r3);
                            const uint32_t a0 = e4m3x2_lo_to_f16x2(r0);
                            const uint32_t a1 = e4m3x2_lo_to_f16x2(r1);
                            const uint32_t a2 = e4m3x2_hi_to_f16x2(r0);
                            const uint32_t a3 = e4m3x2_hi_to_f16x2(r1);
                            const uint32_t b0 = e4m3x2_lo_to_f16x2(r2);
                            const uint32_t b1 = e4m3x2_lo_to_f16x2(r3);
                            const uint32_t b2 = e4m3x2_hi_to_f16x2(r2);
                            const uint32_t b3 = e4m3x2_hi_to_f16x2(r3);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                mma_f16_16816(sc[mt][nt], a0, a1, a2, a3, qf[2 * kp][nt][0],
                                              qf[2 * kp][nt][1]);
                                mma_f16_16816(sc2[mt][nt], b0, b1, b2, b3, qf[2 * kp + 1][nt][0],
                                              qf[2 * kp + 1][nt][1]);
                            }
                        }
                    }
                } else {
#pragma unroll
                for (int mt = 0; mt < S::MT; ++mt) {
                    const int t = mt * 16 + (mi & 1) * 8 + rr;
#pragma unroll
                    for (int kk = 0; kk < S::KD; ++kk) {
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4(kbase + swz<BS>(kk >> 2, t, (kk & 3) * 2 + (mi >> 1)), a0, a1,
                                a2, a3);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            if (kk & 1)
                                mma_bf16_16816(sc2[mt][nt], a0, a1, a2, a3, qf[kk][nt][0],
                                               qf[kk][nt][1]);
                            else
                                mma_bf16_16816(sc[mt][nt], a0, a1, a2, a3, qf[kk][nt][0],
                                               qf[kk][nt][1]);
                        }
                    }
                }
                }
#pragma unroll
                for (int mt = 0; mt < S::MT; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int c = 0; c < 4; ++c) sc[mt][nt][c] += sc2[mt][nt][c];
            }
            // ---- online softmax ----
            // The scores stay unscaled: max(scale * s) = scale * max(s) for the positive
            // scale, and the weights are exp2(fma(s, scale, -m)). Only the last pages of a
            // segment can be partial; a column's keys past its row's causal end become
            // -inf there (the rows of a group end one key apart).
            if constexpr (RG) {
                const int32_t last_keys = cc.kv_len - cc.pp * BS;  // the group's last row, this page
                if (last_keys - (cc.nr - 1) < BS) {  // warp-uniform
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const int lim0 = last_keys - moff[nt][0], lim1 = last_keys - moff[nt][1];
#pragma unroll
                        for (int mt = 0; mt < S::MT; ++mt) {
                            const int t0 = mt * 16 + gl, t1 = t0 + 8;
                            float* c = sc[mt][nt];
                            if (t0 >= lim0) c[0] = -INFINITY;
                            if (t0 >= lim1) c[1] = -INFINITY;
                            if (t1 >= lim0) c[2] = -INFINITY;
                            if (t1 >= lim1) c[3] = -INFINITY;
                        }
                    }
                }
            } else if (nvalid < BS) {  // warp-uniform
#pragma unroll
                for (int mt = 0; mt < S::MT; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const int t0 = mt * 16 + gl, t1 = t0 + 8;
                        float* c = sc[mt][nt];
                        if (t0 >= nvalid) c[0] = c[1] = -INFINITY;
                        if (t1 >= nvalid) c[2] = c[3] = -INFINITY;
                    }
            }
            float corr[NT][2], msafe[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int mt = 0; mt < S::MT; ++mt) {
                    const float* c = sc[mt][nt];
                    mx0 = fmaxf(mx0, fmaxf(c[0], c[2]));
                    mx1 = fmaxf(mx1, fmaxf(c[1], c[3]));
                }
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                }
                const float mn0 = fmaxf(m_run[nt][0], mx0 * sl2p);
                const float mn1 = fmaxf(m_run[nt][1], mx1 * sl2p);
                // a column with no key yet (a group row whose keys all lie on later
                // pages of a backward walk) keeps m = -inf: its weights and factor
                // are taken against 0, so that they are 0 and never NaN
                msafe[nt][0] = (RG && mn0 == -INFINITY) ? 0.f : mn0;
                msafe[nt][1] = (RG && mn1 == -INFINITY) ? 0.f : mn1;
                corr[nt][0] = exp2_approx(m_run[nt][0] - msafe[nt][0]);
                corr[nt][1] = exp2_approx(m_run[nt][1] - msafe[nt][1]);
                m_run[nt][0] = mn0;
                m_run[nt][1] = mn1;
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (corr[nt][0] != 1.f || corr[nt][1] != 1.f) {
#pragma unroll
                    for (int md = 0; md < S::KD; ++md) {
                        o[md][nt][0] *= corr[nt][0];
                        o[md][nt][1] *= corr[nt][1];
                        o[md][nt][2] *= corr[nt][0];
                        o[md][nt][3] *= corr[nt][1];
                    }
                }
                l_part[nt][0] *= corr[nt][0];
                l_part[nt][1] *= corr[nt][1];
            }
            // ---- O^T += V^T P^T ----
            if constexpr (F8) {
                // weights p * vr in f16 for all 16-token tiles; the row sums take p
                uint32_t pb[S::MT][NT][2];
#pragma unroll
                for (int kt = 0; kt < S::MT; ++kt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const float* c = sc[kt][nt];
                        const float p0 = exp2_approx(fmaf(c[0], sl2p, -msafe[nt][0]));
                        const float p1 = exp2_approx(fmaf(c[1], sl2p, -msafe[nt][1]));
                        const float p2 = exp2_approx(fmaf(c[2], sl2p, -msafe[nt][0]));
                        const float p3 = exp2_approx(fmaf(c[3], sl2p, -msafe[nt][1]));
                        l_part[nt][0] += p0 + p2;
                        l_part[nt][1] += p1 + p3;
                        pb[kt][nt][0] = movmatrix_trans(pack_f16x2(p0 * vr, p1 * vr));
                        pb[kt][nt][1] = movmatrix_trans(pack_f16x2(p2 * vr, p3 * vr));
                    }
                // ldmatrix.trans over 16-byte rows hands a lane head dims (2gl, 2gl + 1)
                // of tokens (2tq, 2tq + 1): A-operand row gl takes head dim 2gl and
                // row gl + 8 head dim 2gl + 1 of each 16-wide step.
                const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
                for (int mp = 0; mp < S::KD / 2; ++mp) {
#pragma unroll
                    for (int kt = 0; kt < S::MT; ++kt) {
                        const int t = kt * 16 + (mi & 1) * 8 + rr;
                        const int ch = 2 * mp + (mi >> 1);
                        uint32_t r0, r1, r2, r3;
                        ldsm_x4_trans(vbase + swz<BS>(ch >> 3, t, ch & 7), r0, r1, r2, r3);
                        // bytes (b3 b2 b1 b0) -> (b3 b1 b2 b0): head dim 2gl of both
                        // tokens in the low half, head dim 2gl + 1 in the high half
                        const uint32_t u0 = __byte_perm(r0, 0u, 0x3120u);
                        const uint32_t u1 = __byte_perm(r1, 0u, 0x3120u);
                        const uint32_t u2 = __byte_perm(r2, 0u, 0x3120u);
                        const uint32_t u3 = __byte_perm(r3, 0u, 0x3120u);
                        const uint32_t a0 = e4m3x2_lo_to_f16x2(u0);
                        const uint32_t a1 = e4m3x2_hi_to_f16x2(u0);
                        const uint32_t a2 = e4m3x2_lo_to_f16x2(u1);
                        const uint32_t a3 = e4m3x2_hi_to_f16x2(u1);
                        const uint32_t b0 = e4m3x2_lo_to_f16x2(u2);
                        const uint32_t b1 = e4m3x2_hi_to_f16x2(u2);
                        const uint32_t b2 = e4m3x2_lo_to_f16x2(u3);
                        const uint32_t b3 = e4m3x2_hi_to_f16x2(u3);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            mma_f16_16816(o[2 * mp][nt], a0, a1, a2, a3, pb[kt][nt][0],
                                          pb[kt][nt][1]);
                            mma_f16_16816(o[2 * mp + 1][nt], b0, b1, b2, b3, pb[kt][nt][0],
                                          pb[kt][nt][1]);
                        }
                    }
                }
            } else
#pragma unroll
            for (int kt = 0; kt < S::MT; ++kt) {
                uint32_t pb[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float* c = sc[kt][nt];
                    const uint32_t lo = pack_bf16x2(exp2_approx(fmaf(c[0], sl2p, -msafe[nt][0])),
                                                    exp2_approx(fmaf(c[1], sl2p, -msafe[nt][1])));
                    const uint32_t hi = pack_bf16x2(exp2_approx(fmaf(c[2], sl2p, -msafe[nt][0])),
                                                    exp2_approx(fmaf(c[3], sl2p, -msafe[nt][1])));
                    // row sums use exactly the rounded weights fed to the mma
                    l_part[nt][0] += bf16lo_to_f32(lo) + bf16lo_to_f32(hi);
                    l_part[nt][1] += bf16hi_to_f32(lo) + bf16hi_to_f32(hi);
                    pb[nt][0] = movmatrix_trans(lo);
                    pb[nt][1] = movmatrix_trans(hi);
                }
                const int mi = lane >> 3, rr = lane & 7;
                const int t = kt * 16 + (mi >> 1) * 8 + rr;
#pragma unroll
                for (int md = 0; md < S::KD; ++md) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_trans(vbase + swz<BS>(md >> 2, t, (md & 3) * 2 + (mi & 1)), a0, a1,
                                  a2, a3);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_bf16_16816(o[md][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
                }
            }
        }
        // the stage is free once every warp reading it is done (both of a pair)
        if constexpr (PR) pair_sync(pair_bar);
        else __syncwarp();
        if (lane == 0 && leader && i + STAGES < n_my) {
            issue(i + STAGES);
            if (i + STAGES + 1 < n_my) fetch_blk();
        }

        if (cc.pp == (rev ? 0 : cc.pages - 1) || i == n_my - 1) {  // segment or slice done
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    l_part[nt][0] += __shfl_xor_sync(0xffffffffu, l_part[nt][0], off);
                    l_part[nt][1] += __shfl_xor_sync(0xffffffffu, l_part[nt][1], off);
                }
            const int64_t s0 = cc.seg_start, s1 = cc.seg_start + cc.pages;
            const int nvh = RG ? cc.nr * p.G : p.G;  // virtual heads of the group (row-major over its rows)
            if (s0 >= my_lo && s1 <= my_hi) {
                // whole segment in this worker: final output
                __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int h = c8 + nt * 8 + 2 * tq + e;
                        // a group row without any key (seq_len below its request's rows)
                        // is zero-filled and flagged above: never written here
                        if (h >= nvh || (RG && l_part[nt][e] == 0.f)) continue;
                        const float inv = (F8 ? vref : 1.f) / l_part[nt][e];
                        const int hr = RG ? h / p.G : 0;
                        __nv_bfloat16* dst =
                            outp + ((static_cast<int64_t>(cc.n) + hr) * p.H_q + cc.g * p.G + (h - hr * p.G)) * D;
#pragma unroll
                        for (int md = 0; md < S::KD; ++md) {
                            dst[drow(md, 0)] = __float2bfloat16_rn(o[md][nt][e] * inv);
                            dst[drow(md, 1)] = __float2bfloat16_rn(o[md][nt][2 + e] * inv);
                        }
                    }
            } else {
                const int slot = s0 < my_lo ? 0 : 1;
                // A piece flushed at the end of the slice goes to this warp's
                // ring, idle from here on; the one flushed mid-stream (the
                // first segment walked: it began before the slice and ends
                // inside it, so its slot is 0) goes to the workspace, where
                // the combine reads it.
                const bool at_end = (i == n_my - 1);
                float* dst_o;
                float2* dst_ml;
                if (at_end) {
                    dst_o = reinterpret_cast<float*>(wbuf + slot * piece_bytes);
                    dst_ml = reinterpret_cast<float2*>(dst_o + p.vhs * D);
                } else {
                    const int64_t piece = static_cast<int64_t>(wid) * p.vhs;
                    dst_o = ws.w_o + piece * D;
                    dst_ml = ws.w_ml + piece;
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int h = c8 + nt * 8 + 2 * tq + e;
                        if (h >= nvh) continue;
                        float* dst = dst_o + h * D;
                        const float of = F8 ? vref : 1.f;  // partials in true units
#pragma unroll
                        for (int md = 0; md < S::KD; ++md) {
                            dst[drow(md, 0)] = o[md][nt][e] * of;
                            dst[drow(md, 1)] = o[md][nt][2 + e] * of;
                        }
                        if (gl == 0) dst_ml[h] = make_float2(m_run[nt][e], l_part[nt][e]);
                    }
                if (lane == 0 && leader) {
                    hdr[wk][slot].s0 = s0;
                    hdr[wk][slot].s1 = s1;
                    hdr[wk][slot].n = cc.n;
                    hdr[wk][slot].g = cc.g;
                    hdr[wk][slot].nr = cc.nr;
                    hdr[wk][slot].o = dst_o;
                    hdr[wk][slot].ml = dst_ml;
                    hdr[wk][slot].valid = 1;
                }
            }
            reset_state();
        }
        step(cc);
    }

    if (aborted) {
        // drain the copies of this worker still in flight before the CTA exits
        const int issued = n_my < consumed + STAGES ? n_my : consumed + STAGES;
        for (int i = consumed; i < issued; ++i)
            (void)mbar_wait_bounded(wbar + (i % STAGES), (i / STAGES) & 1, kWaitLimitNs);
        if (lane == 0) {
            set_err(p.err, YOCO_DEVERR_TIMEOUT);
            atomicExch(&abort_flag, 1);
        }
    }
    __syncthreads();  // pieces and headers are visible to the whole CTA
    if (abort_flag) return;

    // ---- combine the pieces of each segment this CTA holds, in worker order ----
    // A group is the run of valid pieces (worker, then slot order) of one
    // segment. Every thread walks the groups itself and derives the scale
    // factors it needs, so the combine has no barrier and no serial step: it
    // runs once per launch, right after streaming, with a cold instruction
    // cache and L2 still busy with the other SMs' streams, where each barrier
    // or dependent step costs far more than the arithmetic. Groups of up to 8
    // heads (one tile) take one four-element vector per thread and step; wider
    // groups lay the threads out head-major, each taking one head and every
    // tph-th vector of it, so the factors are derived once per head, not once
    // per vector.
    constexpr int MAXE = 2 * WK;
    constexpr int D4 = D / 4;  // four-element vectors per head
    __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(p.out);
    const int VS = p.vhs;       // virtual heads per partial slot
    // two tiles: threads per (virtual) head, and this thread's head (past the
    // segment's heads: idle)
    const int tph = static_cast<int>(blockDim.x) / (RG ? VS : p.G);
    const int ch = static_cast<int>(threadIdx.x) / tph;
    int e0 = 0;
    for (;;) {
        while (e0 < MAXE && !hdr[e0 >> 1][e0 & 1].valid) ++e0;
        if (e0 >= MAXE || (NTG != 1 && !RG && ch >= p.G)) break;
        const int64_t s0 = hdr[e0 >> 1][e0 & 1].s0, s1 = hdr[e0 >> 1][e0 & 1].s1;
        const int32_t gn = hdr[e0 >> 1][e0 & 1].n, gg = hdr[e0 >> 1][e0 & 1].g;
        const int32_t gnr = hdr[e0 >> 1][e0 & 1].nr;
        int e1 = e0 + 1;  // one past the group (entries in between may be invalid)
        while (e1 < MAXE && (!hdr[e1 >> 1][e1 & 1].valid || hdr[e1 >> 1][e1 & 1].s0 == s0)) ++e1;
        if (NTG != 1 && RG && ch >= gnr * p.G) {  // no head of this thread in the group
            e0 = e1;
            continue;
        }
        const bool whole = s0 >= cta_lo && s1 <= cta_hi;
        if constexpr (NTG == 1) {
            const int cslot = s0 < cta_lo ? 0 : 1;
            // groups of rows (one 8-head tile) are laid out row-major: virtual head h
            // is head h % G of row gn + h / G
            const int nvec = gnr * p.G * D4;  // four-element vectors of the segment's output
            for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
                const int h = (v * 4) / D;
                float M = -INFINITY;
#pragma unroll 4
                for (int e = e0; e < e1; ++e) {
                    const PieceHdr& X = hdr[e >> 1][e & 1];
                    if (X.valid) M = fmaxf(M, X.ml[h].x);
                }
                float L = 0.f;
                float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
                for (int e = e0; e < e1; ++e) {
                    const PieceHdr& X = hdr[e >> 1][e & 1];
                    if (!X.valid) continue;
                    const float2 ml = X.ml[h];
                    const float4 x = reinterpret_cast<const float4*>(X.o)[v];
                    const float f = ml.x != -INFINITY ? exp2_approx(ml.x - M) : 0.f;
                    L += ml.y * f;
                    O.x += x.x * f;
                    O.y += x.y * f;
                    O.z += x.z * f;
                    O.w += x.w * f;
                }
                if (whole) {
                    if (RG && L == 0.f) continue;  // a group row without keys: zero-filled above
                    const float inv = 1.f / L;
                    const int hr = RG ? h / p.G : 0;
                    __nv_bfloat16* dst = outp + ((static_cast<int64_t>(gn) + hr) * p.H_q + gg * p.G +
                                                 (h - hr * p.G)) * D + (v * 4 - h * D);
                    reinterpret_cast<__nv_bfloat162*>(dst)[0] = __floats2bfloat162_rn(O.x * inv, O.y * inv);
                    reinterpret_cast<__nv_bfloat162*>(dst)[1] = __floats2bfloat162_rn(O.z * inv, O.w * inv);
                } else {
                    const int64_t cp = (static_cast<int64_t>(blockIdx.x) * 2 + cslot) * VS + h;
                    reinterpret_cast<float4*>(ws.c_o + cp * D)[(v * 4 - h * D) / 4] = O;
                    if (v * 4 - h * D == 0) ws.c_ml[cp] = make_float2(M, L);
                }
            }
        } else {
            const int cr = static_cast<int>(threadIdx.x) - ch * tph;
            const int h = ch;
            float M = -INFINITY;
#pragma unroll 4
            for (int e = e0; e < e1; ++e) {
                const PieceHdr& X = hdr[e >> 1][e & 1];
                if (X.valid) M = fmaxf(M, X.ml[h].x);
            }
            const int64_t cp = (static_cast<int64_t>(blockIdx.x) * 2 + (s0 < cta_lo ? 0 : 1)) * VS + h;
            const int hr = RG ? h / p.G : 0;  // virtual head h: head h % G of row gn + h / G
            __nv_bfloat16* dsth =
                outp + ((static_cast<int64_t>(gn) + hr) * p.H_q + gg * p.G + (h - hr * p.G)) * D;
            for (int c0 = cr; c0 < D4; c0 += 4 * tph) {  // up to four vectors per pass
                float4 O[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) O[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                float L = 0.f;
#pragma unroll 2
                for (int e = e0; e < e1; ++e) {
                    const PieceHdr& X = hdr[e >> 1][e & 1];
                    if (!X.valid) continue;
                    const float2 ml = X.ml[h];
                    const float f = ml.x != -INFINITY ? exp2_approx(ml.x - M) : 0.f;
                    L += ml.y * f;
                    const float4* xo = reinterpret_cast<const float4*>(X.o) + h * D4;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        if (c0 + u * tph < D4) {
                            const float4 x = xo[c0 + u * tph];
                            O[u].x += x.x * f;
                            O[u].y += x.y * f;
                            O[u].z += x.z * f;
                            O[u].w += x.w * f;
                        }
                    }
                }
                const float inv = 1.f / L;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int j = c0 + u * tph;
                    if (j >= D4) continue;
                    if (whole) {
                        if (RG && L == 0.f) continue;  // a group row without keys: zero-filled above
                        __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(dsth + j * 4);
                        dst[0] = __floats2bfloat162_rn(O[u].x * inv, O[u].y * inv);
                        dst[1] = __floats2bfloat162_rn(O[u].z * inv, O[u].w * inv);
                    } else {
                        reinterpret_cast<float4*>(ws.c_o + cp * D)[j] = O[u];
                    }
                }
                if (!whole && c0 == 0) ws.c_ml[cp] = make_float2(M, L);
            }
        }
        e0 = e1;
    }
    __syncthreads();  // every CTA-level partial of this CTA has been written
    // The next kernel in the stream (the next layer) may be scheduled now: it
    // can only take an SM as this grid's CTAs exit, and it waits for the whole
    // grid before it touches the workspace, queries or outputs.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    cross_cta_merge<D, RG>(p, ws, cta_hdr, reinterpret_cast<float*>(smem));
}

// One-time (per device) setting of a kernel's dynamic shared memory limit.
// `done` must be distinct per kernel: callers keep it in a function that is
// itself instantiated per kernel.
template <typename K>
cudaError_t ensure_smem_attr(K kernel, int bytes, unsigned long long& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0;
    if (bit && (__atomic_load_n(&done, __ATOMIC_ACQUIRE) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) __atomic_fetch_or(&done, bit, __ATOMIC_RELEASE);
    return e;
}

// Two-tile walks (groups over 8 heads, or rows grouped 16 wide) run as warp
// pairs at these head dims, except the fused decode step (one warp per ring),
// where a pair kernel has at most 8 warps (registers for the one-tile walk).
template <int D, int BS, bool F8>
constexpr bool tc_pairs() {
    return (D == 256 ? YOCO_TC_PAIRS256 != 0 : D == 128 ? YOCO_TC_PAIRS128 != 0 : false) &&
           TcShape<D, BS, F8, 1, true>::NW <= 8;
}

template <int D, int BS, int NT, bool F8, bool PR>
cudaError_t launch_one(const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p, int sms,
                       cudaStream_t s) {
    using S = TcShape<D, BS, F8, NT, PR>;
    static unsigned long long smem_fwd = 0, smem_rev = 0, smem_fuse = 0;  // one per kernel
    static unsigned long long smem_gfwd = 0, smem_grev = 0;
    const int ctas = tc_ctas(sms);
    // the cross-CTA merge keeps its tables in the (then idle) ring
    if ((16 + 2 * merge_scratch_floats(ctas, 16, D)) * 4 > S::SMEM - 1024)
        return cudaErrorInvalidConfiguration;
    const bool fuse = p.k_new != nullptr, grouped = p.rg > 1;
    if (grouped && fuse) return cudaErrorInvalidConfiguration;
    if (PR && fuse) return cudaErrorInvalidConfiguration;  // the fused step runs one warp per ring
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(S::NW * 32);
    cfg.stream = s;
    cfg.attrs = attr;
    cudaError_t e;
    if (!p.planned) {
        // The step's plan (one warp per worker). It may start while the
        // previous kernel drains when the caller allows the overlap (it reads
        // only the metadata before its dependency wait); the attention launch
        // below reads the plan at its very start, so it is an ordinary (fully
        // ordered) launch.
        cfg.dynamicSmemBytes = 0;
        cfg.blockDim = dim3(S::WK * 32);
        cfg.numAttrs = p.overlap ? 1 : 0;
        e = cudaLaunchKernelEx(&cfg, attn_tc_plan<S::WK, S::STAGES, D, BS>, p);
        if (e != cudaSuccess || p.plan_only) return e;
        cfg.blockDim = dim3(S::NW * 32);
    }
    // row groups and warp pairs: kernels of their own. Where two-tile walks run
    // as warp pairs, a one-warp two-tile kernel serves the fused step alone.
    using K = void (*)(CUtensorMap, CUtensorMap, AttnParams);
    K kernel;
    if constexpr (!PR && NT == 2 && tc_pairs<D, BS, F8>()) {
        if (!fuse) return cudaErrorInvalidConfiguration;
        kernel = attn_tc_persistent<D, BS, NT, false, F8, true, false, false>;
    } else if constexpr (PR) {
        kernel = grouped ? (p.reverse ? attn_tc_persistent<D, BS, NT, true, F8, false, true, true>
                                      : attn_tc_persistent<D, BS, NT, false, F8, false, true, true>)
                         : (p.reverse ? attn_tc_persistent<D, BS, NT, true, F8, false, false, true>
                                      : attn_tc_persistent<D, BS, NT, false, F8, false, false, true>);
    } else {
        kernel = fuse ? attn_tc_persistent<D, BS, NT, false, F8, true, false, false>
                 : grouped ? (p.reverse ? attn_tc_persistent<D, BS, NT, true, F8, false, true, false>
                                        : attn_tc_persistent<D, BS, NT, false, F8, false, true, false>)
                           : (p.reverse ? attn_tc_persistent<D, BS, NT, true, F8, false, false, false>
                                        : attn_tc_persistent<D, BS, NT, false, F8, false, false, false>);
    }
    unsigned long long& done = fuse ? smem_fuse
                               : grouped ? (p.reverse ? smem_grev : smem_gfwd)
                                         : (p.reverse ? smem_rev : smem_fwd);
    e = ensure_smem_attr(kernel, S::SMEM, done);
    if (e != cudaSuccess) return e;
    // With a plan made earlier and the caller's leave, the launch is a
    // programmatic dependent of the kernel before it (for example the previous
    // layer): its prologue (plan record, first page copies) overlaps that
    // kernel's end, and it waits before touching queries, outputs or the
    // workspace.
    cfg.dynamicSmemBytes = S::SMEM;
    cfg.numAttrs = (p.planned && p.overlap) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, mk, mv, p);
}

template <int D, int BS, bool F8>
cudaError_t launch_bs(const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p, int sms,
                      cudaStream_t s) {
    const bool wide = p.vhs > 8;  // two 8-head tiles: a group over 8, or 16 virtual heads
    if constexpr (tc_pairs<D, BS, F8>()) {
        if (wide && p.k_new == nullptr) return launch_one<D, BS, 1, F8, true>(mk, mv, p, sms, s);
    }
    return wide ? launch_one<D, BS, 2, F8, false>(mk, mv, p, sms, s)
                : launch_one<D, BS, 1, F8, false>(mk, mv, p, sms, s);
}

template <int D, bool F8>
cudaError_t launch_d(const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p, int BS,
                     int sms, cudaStream_t s) {
    return BS == 16 ? launch_bs<D, 16, F8>(mk, mv, p, sms, s) : launch_bs<D, 32, F8>(mk, mv, p, sms, s);
}

}  // namespace
}  // namespace yoco
