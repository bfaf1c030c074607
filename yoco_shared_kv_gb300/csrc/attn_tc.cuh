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
// owns pages [P c / C, P (c+1) / C) and each of its NW warps owns an equal
// contiguous slice of that, streamed through the warp's own TMA ring. Every
// worker therefore moves the same number of bytes, whatever the length mix,
// and the ring never drains between segments.
//   - A segment that lies inside one warp's slice is finished in registers
//     and written straight to `out`.
//   - A segment cut by a warp boundary leaves a partial (m, l, o) per piece;
//     at the end of the kernel the CTA combines the pieces of each segment
//     it holds, writing `out` when the CTA holds the whole segment and a
//     CTA-level partial otherwise.
//   - A segment cut by a CTA boundary is finished by attn_tc_merge, which
//     combines the CTA partials in CTA order.
// Every combine runs in a fixed order that depends only on logical page
// indices, so the output is bit-identical under any physical page placement.
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
// tunables; the defaults fill about 192 KiB of shared memory).
#ifndef YOCO_TC_NW16
#define YOCO_TC_NW16 4
#endif
#ifndef YOCO_TC_ST16
#define YOCO_TC_ST16 3
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
// NT: 8-head tiles of the group (1 for groups up to 8, else 2).
template <int D, int BS, bool F8 = false, int NT = 2>
struct TcShape {
    static constexpr int ESZ = F8 ? 1 : 2;                // bytes per cached element
    static constexpr int PAGE_BYTES = BS * D * ESZ;       // K (or V) of one page, one kv head
    static constexpr int STAGE_BYTES = 2 * PAGE_BYTES;    // K + V
    // a warp's two end-of-slice pieces at the largest group of this NT
    static constexpr int PIECE_PAIR = 2 * (8 * NT * (D * 4 + 8) + 16);
    // the most warps (8, 4, 2) whose ring share holds two stages and the two pieces
    static constexpr int F8_FITS8 =
        PIECE_PAIR <= YOCO_TC_F8_RING / 8 && 2 * STAGE_BYTES <= YOCO_TC_F8_RING / 8;
    static constexpr int F8_FITS4 =
        PIECE_PAIR <= YOCO_TC_F8_RING / 4 && 2 * STAGE_BYTES <= YOCO_TC_F8_RING / 4;
    static constexpr int F8_NW =
        YOCO_TC_F8_NW > 0 ? YOCO_TC_F8_NW : (F8_FITS8 ? 8 : (F8_FITS4 ? 4 : 2));
    static constexpr int NW =
        F8 ? F8_NW : (STAGE_BYTES <= 8192 ? 8 : (STAGE_BYTES <= 16384 ? YOCO_TC_NW16 : 2));
    // e4m3 pages are small: deepen the ring to keep ~192 KiB in flight per SM
    static constexpr int F8_STAGES = YOCO_TC_F8_RING / F8_NW / STAGE_BYTES;
    static constexpr int STAGES =
        F8 ? (F8_STAGES < 2 ? 2 : F8_STAGES) : (STAGE_BYTES == 16384 ? YOCO_TC_ST16 : 3);
    static constexpr int SUBE = 128 / ESZ;  // elements per 128-byte row of a sub-tile
    static constexpr int KSUB = D / SUBE;   // 128-byte swizzled sub-tiles per row
    static constexpr int SUB_BYTES = BS * 128;
    static constexpr int MT = BS / 16;   // 16-token tiles per page
    static constexpr int KD = D / 16;    // 16-wide steps along head_dim
    static constexpr int SMEM = NW * STAGES * STAGE_BYTES + 1024;
    static_assert(SMEM <= 200 * 1024, "the rings must leave room for static shared memory");
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

// Pages (all kv heads) of request r's cross rows below max_rows.
__device__ __forceinline__ int64_t req_pages(const AttnParams& p, int32_t r, int32_t cap) {
    const int32_t c0 = __ldg(p.cqsl + r), c1 = __ldg(p.cqsl + r + 1);
    const int32_t k = c1 - c0, hi = min(c1, p.max_rows), seq = __ldg(p.seq_lens + r);
    int64_t s = 0;
    for (int32_t n = c0; n < hi; ++n) s += row_pages(seq - k + (n - c0) + 1, cap, p.block_size);
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
    int32_t req, n, g, pp, kv_len, pages;
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
            const int32_t k = c1 - c0, seq = __ldg(p.seq_lens + req);
            for (int32_t n = c0; n < c1 && n < p.max_rows; ++n) {
                const int32_t kv = seq - k + (n - c0) + 1;
                const int32_t pg = row_pages(kv, cap, p.block_size);
                const int64_t seg_pages = static_cast<int64_t>(pg) * p.H_kv;
                if (x < off + seg_pages) {
                    const int64_t rel = x - off;
                    c.req = req;
                    c.n = n;
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

// Next page in the flattened order (skips rows without keys).
__device__ __forceinline__ void advance(const AttnParams& p, Cursor& c, int32_t cap) {
    if (++c.pp < c.pages) return;
    c.seg_start += c.pages;
    c.pp = 0;
    if (++c.g < p.H_kv) return;
    c.g = 0;
    for (;;) {
        if (++c.n >= p.max_rows) return;
        while (c.req + 1 < p.num_reqs && __ldg(p.cqsl + c.req + 1) <= c.n) ++c.req;
        const int32_t c0 = __ldg(p.cqsl + c.req), c1 = __ldg(p.cqsl + c.req + 1);
        if (c.n >= c1) return;
        const int32_t kv = __ldg(p.seq_lens + c.req) - (c1 - c0) + (c.n - c0) + 1;
        c.pages = row_pages(kv, cap, p.block_size);
        c.kv_len = min(kv, cap);
        if (c.pages > 0) return;
    }
}

// Previous page in the flattened order (skips rows without keys).
__device__ __forceinline__ void retreat(const AttnParams& p, Cursor& c, int32_t cap) {
    if (--c.pp >= 0) return;
    if (--c.g >= 0) {  // same row, previous kv head
        c.pp = c.pages - 1;
        c.seg_start -= c.pages;
        return;
    }
    for (;;) {
        if (--c.n < 0) return;
        while (c.req > 0 && __ldg(p.cqsl + c.req) > c.n) --c.req;
        const int32_t c0 = __ldg(p.cqsl + c.req), c1 = __ldg(p.cqsl + c.req + 1);
        const int32_t kv = __ldg(p.seq_lens + c.req) - (c1 - c0) + (c.n - c0) + 1;
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

// Most CTAs one merge can span (the grid has one CTA per SM).
constexpr int kMaxMergePieces = 1024;

struct PieceHdr {
    int64_t s0, s1;    // segment [first page, end) in the flattened order
    const float* o;    // [G][D] partial output: in the warp's ring or in the workspace
    const float2* ml;  // [G] (m, l)
    int32_t n, g;
    int32_t valid;
};

// The segments holding a CTA's first and last page, as seen by that CTA
// (read by the merge kernel, so it needs no scan of the metadata itself).
struct CtaHdr {
    int64_t P;       // pages of the launch
    int64_t a0, a1;  // segment of the first page [first, end); a0 < 0: slice starts past the end
    int64_t b0, b1;  // segment of the last page; b0 < 0: empty slice
    int32_t an, ag;  // (row, kv head) of segment a
    int32_t bn, bg;  // (row, kv head) of segment b
};

// Workspace carve-up: [W + C][2][G][D] partial outputs (warp pieces, then CTA
// pieces), [W + C][2][G] (m, l), then one header per CTA.
struct TcWs {
    float* w_o;
    float* c_o;
    float2* w_ml;
    float2* c_ml;
    CtaHdr* hdr;
};

__host__ __device__ __forceinline__ int64_t tc_pieces(int64_t ctas, int nw, int G) {
    return (ctas * nw + ctas) * 2 * G;
}

__device__ __forceinline__ TcWs tc_ws(const AttnParams& p, int ctas, int nw, int D) {
    TcWs w;
    const int64_t per = 2ll * p.G;  // pieces per worker (first / last segment) x heads
    const int64_t W = static_cast<int64_t>(ctas) * nw;
    w.w_o = p.ws_o;
    w.c_o = p.ws_o + W * per * D;
    w.w_ml = p.ws_ml;
    w.c_ml = p.ws_ml + W * per;
    w.hdr = reinterpret_cast<CtaHdr*>(p.ws_ml + tc_pieces(ctas, nw, p.G));
    return w;
}

// --------------------------------------------------------------- kernel

// FUSE: fused decode step (append this step's tokens, patch them into the
// copied pages); instantiated with REV = false only.
template <int D, int BS, int NT, bool REV, bool F8, bool FUSE>
__global__ void __launch_bounds__(TcShape<D, BS, F8, NT>::NW * 32, 1)
    attn_tc_persistent(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
    using S = TcShape<D, BS, F8, NT>;
    constexpr int NW = S::NW, STAGES = S::STAGES;
    static_assert(S::PIECE_PAIR <= STAGES * S::STAGE_BYTES,
                  "a warp's two end-of-slice pieces must fit in its ring");
    static_assert(!F8 || D % 128 == 0, "e4m3 pages need 128-byte rows");
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[NW * STAGES];
    __shared__ int32_t stage_blk[NW * STAGES];  // physical page of each stage (-1: invalid)
    // e4m3: the page's scale record {k_scale, v_scale, -, -}, copied with the page
    __shared__ __align__(16) float4 stage_scale[F8 ? NW * STAGES : 1];
    __shared__ PieceHdr hdr[NW][2];
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gl = lane >> 2, tq = lane & 3;  // mma fragment row group / column pair
    if (threadIdx.x == 0) abort_flag = launch_aborted(p) ? 1 : 0;
    if (lane == 0) {
        for (int i = 0; i < STAGES; ++i) mbar_init(&bars[warp * STAGES + i], 1);
        fence_mbar_init();
        hdr[warp][0].valid = hdr[warp][1].valid = 0;
    }
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    __syncthreads();
    if (abort_flag) return;

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const int64_t cap64 = static_cast<int64_t>(p.max_blocks) * BS;
    const int32_t cap = cap64 > 0x7fffffff ? 0x7fffffff : static_cast<int32_t>(cap64);
    const int64_t P = total_pages(p, lane, cap);
    const int64_t C = gridDim.x;
    const int64_t cta_lo = P * blockIdx.x / C, cta_hi = P * (blockIdx.x + 1) / C;
    const int64_t my_lo = cta_lo + (cta_hi - cta_lo) * warp / NW;
    const int64_t my_hi = cta_lo + (cta_hi - cta_lo) * (warp + 1) / NW;
    const int32_t n_my = static_cast<int32_t>(my_hi - my_lo);
    const int32_t wid = blockIdx.x * NW + warp;
    const TcWs ws = tc_ws(p, gridDim.x, NW, D);

    uint8_t* wbuf = smem + warp * STAGES * S::STAGE_BYTES;
    uint64_t* wbar = bars + warp * STAGES;
    // Odd layers may walk each slice backwards (REV): a layer then starts on
    // the pages the previous layer read last, which are still in L2.
    constexpr bool rev = REV;
    auto step = [&](Cursor& c) {
        if (rev) retreat(p, c, cap);
        else advance(p, c, cap);
    };
    Cursor cc;  // page being consumed
    cc.req = -1;
    if (n_my > 0) locate(p, lane, rev ? my_hi - 1 : my_lo, cap, cc);
    // header for the merge kernel: warp 0 finds the segment of page cta_lo,
    // warp 1 the segment of page cta_hi - 1
    int64_t hs0 = -1, hs1 = -1;
    int32_t hn = 0, hg = 0;
    if (warp <= 1) {
        const int64_t x = warp == 0 ? cta_lo : cta_hi - 1;
        const bool any = warp == 0 ? cta_lo < P : cta_hi > cta_lo;
        Cursor h0 = cc;
        if (any && !(warp == 0 && n_my > 0 && !rev)) locate(p, lane, x, cap, h0);
        if (any && h0.req >= 0) {
            hs0 = h0.seg_start;
            hs1 = h0.seg_start + h0.pages;
            hn = h0.n;
            hg = h0.g;
        }
    }
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
        kKeepBytes / (static_cast<int64_t>(gridDim.x) * NW * S::STAGE_BYTES));
    auto issue = [&](int i) {  // lane 0 only; pc is at page i, blk_next its entry
        const int st = i % STAGES;
        uint64_t* bar = wbar + st;
        const int32_t blk = blk_next;
        // published to the consumer lanes by the barrier's release/acquire
        stage_blk[warp * STAGES + st] = (blk < 0 || blk >= p.num_blocks) ? -1 : blk;
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
                bulk_load(&stage_scale[warp * STAGES + st],
                          p.scales + static_cast<int64_t>(blk) * p.H_kv + pc.g, 16, bar);
        }
        step(pc);
        if (i + 1 < n_my) fetch_blk();
    };
    if (lane == 0) {
        if (n_my > 0) fetch_blk();
        const int pro = n_my < STAGES ? n_my : STAGES;
        for (int i = 0; i < pro; ++i) issue(i);
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
    if (lane == 0 && warp <= 1) {
        CtaHdr* hp = ws.hdr + blockIdx.x;
        if (warp == 0) {
            hp->P = P;
            hp->a0 = hs0;
            hp->a1 = hs1;
            hp->an = hn;
            hp->ag = hg;
        } else {
            hp->b0 = hs0;
            hp->b1 = hs1;
            hp->bn = hn;
            hp->bg = hg;
        }
    }

    uint32_t qf[S::KD][NT][2];
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
    auto load_q = [&](int32_t n, int32_t g) {
        const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(p.q) +
                                    (static_cast<int64_t>(n) * p.H_q + g * p.G) * D;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int h = nt * 8 + gl;
            const bool ok = h < p.G;
            if constexpr (F8) {
                const uint2* src = reinterpret_cast<const uint2*>(qrow + (ok ? h : 0) * D);
#pragma unroll
                for (int kk = 0; kk < S::KD; ++kk) {
                    const uint2 v = ok ? __ldg(src + kk * 4 + tq) : make_uint2(0u, 0u);
                    qf[kk][nt][0] = pack_f16x2(bf16lo_to_f32(v.x), bf16hi_to_f32(v.x));
                    qf[kk][nt][1] = pack_f16x2(bf16lo_to_f32(v.y), bf16hi_to_f32(v.y));
                }
            } else {
                const uint32_t* src = reinterpret_cast<const uint32_t*>(qrow + (ok ? h : 0) * D);
#pragma unroll
                for (int kk = 0; kk < S::KD; ++kk) {
                    qf[kk][nt][0] = ok ? __ldg(src + kk * 8 + tq) : 0u;
                    qf[kk][nt][1] = ok ? __ldg(src + kk * 8 + 4 + tq) : 0u;
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
    const int piece_bytes = (p.G * (D * 4 + 8) + 15) & ~15;

    for (int i = 0; i < n_my; ++i) {
        if (i == 0 || cc.pp == (rev ? cc.pages - 1 : 0)) {
            load_q(cc.n, cc.g);
            if (fused) load_patch(cc.req, cc.g);
        }
        const int st = i % STAGES;
        if (!mbar_wait_bounded(wbar + st, (i / STAGES) & 1, kWaitLimitNs)) {
            aborted = true;
            break;
        }
        consumed = i + 1;
        if (stage_blk[warp * STAGES + st] >= 0) {
            const uint32_t kbase = smem_u32(wbuf + st * S::STAGE_BYTES);
            const uint32_t vbase = kbase + S::PAGE_BYTES;
            const int32_t nvalid = min(BS, cc.kv_len - cc.pp * BS);
            float sl2p = sl2, vr = 1.f;  // score factor, weight factor of this page
            if constexpr (F8) {
                // codes widen exactly; the page's K scale goes into the score factor
                const float4 sc4 = stage_scale[warp * STAGES + st];
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
                        const float4 sc4 = stage_scale[warp * STAGES + st];
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
                uint8_t* vd = wbuf + st * S::STAGE_BYTES + S::PAGE_BYTES;
                const int nbytes = (BS - nvalid) * 128;
                for (int c = 0; c < S::KSUB; ++c)
                    for (int b = lane * 16; b < nbytes; b += 32 * 16)
                        *reinterpret_cast<uint4*>(vd + c * S::SUB_BYTES + nvalid * 128 + b) =
                            make_uint4(0, 0, 0, 0);
                fence_proxy_async_smem();
                __syncwarp();
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
                if constexpr (F8) {
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
            // scale, and the weights are exp2(fma(s, scale, -m)). Only a segment's last
            // page can be partial; its keys past the causal end become -inf there.
            if (nvalid < BS) {  // warp-uniform
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
            float corr[NT][2];
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
                corr[nt][0] = exp2_approx(m_run[nt][0] - mn0);
                corr[nt][1] = exp2_approx(m_run[nt][1] - mn1);
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
                        const float p0 = exp2_approx(fmaf(c[0], sl2p, -m_run[nt][0]));
                        const float p1 = exp2_approx(fmaf(c[1], sl2p, -m_run[nt][1]));
                        const float p2 = exp2_approx(fmaf(c[2], sl2p, -m_run[nt][0]));
                        const float p3 = exp2_approx(fmaf(c[3], sl2p, -m_run[nt][1]));
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
                    const uint32_t lo = pack_bf16x2(exp2_approx(fmaf(c[0], sl2p, -m_run[nt][0])),
                                                    exp2_approx(fmaf(c[1], sl2p, -m_run[nt][1])));
                    const uint32_t hi = pack_bf16x2(exp2_approx(fmaf(c[2], sl2p, -m_run[nt][0])),
                                                    exp2_approx(fmaf(c[3], sl2p, -m_run[nt][1])));
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
        __syncwarp();
        if (lane == 0 && i + STAGES < n_my) issue(i + STAGES);

        if (cc.pp == (rev ? 0 : cc.pages - 1) || i == n_my - 1) {  // segment or slice done
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    l_part[nt][0] += __shfl_xor_sync(0xffffffffu, l_part[nt][0], off);
                    l_part[nt][1] += __shfl_xor_sync(0xffffffffu, l_part[nt][1], off);
                }
            const int64_t s0 = cc.seg_start, s1 = cc.seg_start + cc.pages;
            const int64_t head0 = static_cast<int64_t>(cc.n) * p.H_q + cc.g * p.G;
            if (s0 >= my_lo && s1 <= my_hi) {
                // whole segment in this warp: final output
                __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int h = nt * 8 + 2 * tq + e;
                        if (h >= p.G) continue;
                        const float inv = (F8 ? vref : 1.f) / l_part[nt][e];
                        __nv_bfloat16* dst = outp + (head0 + h) * D;
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
                // first segment walked) goes to the workspace, where the
                // combine reads it.
                const bool at_end = (i == n_my - 1);
                float* dst_o;
                float2* dst_ml;
                if (at_end) {
                    dst_o = reinterpret_cast<float*>(wbuf + slot * piece_bytes);
                    dst_ml = reinterpret_cast<float2*>(dst_o + p.G * D);
                } else {
                    const int64_t piece = (static_cast<int64_t>(wid) * 2 + slot) * p.G;
                    dst_o = ws.w_o + piece * D;
                    dst_ml = ws.w_ml + piece;
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int h = nt * 8 + 2 * tq + e;
                        if (h >= p.G) continue;
                        float* dst = dst_o + h * D;
                        const float of = F8 ? vref : 1.f;  // partials in true units
#pragma unroll
                        for (int md = 0; md < S::KD; ++md) {
                            dst[drow(md, 0)] = o[md][nt][e] * of;
                            dst[drow(md, 1)] = o[md][nt][2 + e] * of;
                        }
                        if (gl == 0) dst_ml[h] = make_float2(m_run[nt][e], l_part[nt][e]);
                    }
                if (lane == 0) {
                    hdr[warp][slot].s0 = s0;
                    hdr[warp][slot].s1 = s1;
                    hdr[warp][slot].n = cc.n;
                    hdr[warp][slot].g = cc.g;
                    hdr[warp][slot].o = dst_o;
                    hdr[warp][slot].ml = dst_ml;
                    hdr[warp][slot].valid = 1;
                }
            }
            reset_state();
        }
        step(cc);
    }

    if (aborted) {
        // drain this warp's copies still in flight before the CTA exits
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

    // ---- combine the pieces of each segment this CTA holds, in warp order ----
    // A group is the run of valid pieces (warp, then slot order) of one
    // segment. Every thread walks the groups itself and derives the scale
    // factors it needs, so the combine has no barrier and no serial step: it
    // runs once per launch, right after streaming, with a cold instruction
    // cache and L2 still busy with the other SMs' streams, where each barrier
    // or dependent step costs far more than the arithmetic. Groups of up to 8
    // heads (one tile) take one four-element vector per thread and step; wider
    // groups lay the threads out head-major, each taking one head and every
    // tph-th vector of it, so the factors are derived once per head, not once
    // per vector.
    constexpr int MAXE = 2 * NW;
    constexpr int D4 = D / 4;  // four-element vectors per head
    __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(p.out);
    const int tph = static_cast<int>(blockDim.x) / p.G;     // threads per head (G <= 16)
    const int ch = static_cast<int>(threadIdx.x) / tph;     // this thread's head (G or more: idle)
    const int nvec = p.G * D4;  // four-element vectors of a segment's output
    int e0 = 0;
    for (;;) {
        while (e0 < MAXE && !hdr[e0 >> 1][e0 & 1].valid) ++e0;
        if (e0 >= MAXE || (NT != 1 && ch >= p.G)) break;
        const int64_t s0 = hdr[e0 >> 1][e0 & 1].s0, s1 = hdr[e0 >> 1][e0 & 1].s1;
        const int32_t gn = hdr[e0 >> 1][e0 & 1].n, gg = hdr[e0 >> 1][e0 & 1].g;
        int e1 = e0 + 1;  // one past the group (entries in between may be invalid)
        while (e1 < MAXE && (!hdr[e1 >> 1][e1 & 1].valid || hdr[e1 >> 1][e1 & 1].s0 == s0)) ++e1;
        const bool whole = s0 >= cta_lo && s1 <= cta_hi;
        if constexpr (NT == 1) {
            const int cslot = s0 < cta_lo ? 0 : 1;
            const int64_t head0 = static_cast<int64_t>(gn) * p.H_q + gg * p.G;
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
                    const float inv = 1.f / L;
                    __nv_bfloat16* dst = outp + head0 * D + v * 4;
                    reinterpret_cast<__nv_bfloat162*>(dst)[0] = __floats2bfloat162_rn(O.x * inv, O.y * inv);
                    reinterpret_cast<__nv_bfloat162*>(dst)[1] = __floats2bfloat162_rn(O.z * inv, O.w * inv);
                } else {
                    const int64_t cp = (static_cast<int64_t>(blockIdx.x) * 2 + cslot) * p.G + h;
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
            const int64_t cp = (static_cast<int64_t>(blockIdx.x) * 2 + (s0 < cta_lo ? 0 : 1)) * p.G + h;
            __nv_bfloat16* dsth = outp + (static_cast<int64_t>(gn) * p.H_q + gg * p.G + h) * D;
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
    // the merge kernel may be scheduled now (it waits for this grid to finish);
    // triggering only here keeps its waiting CTAs off the SM during the combine
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Finishes every segment cut by a CTA boundary from the CTA-level partials
// (rows with no key are zero-filled by the split kernel). Grid: one CTA per
// split-kernel CTA.
// Each CTA spanned by a cut segment takes an equal share of that segment's
// G x D outputs, so a long segment's merge spreads over all of its CTAs. A
// CTA shares at most two segments (those of its first and last page); the
// two halves of the CTA work on them at the same time. Pieces are combined
// in CTA order.
constexpr int kMergeThreads = 256;
constexpr int kMergeHalf = kMergeThreads / 2;
constexpr int kMergeRegPieces = 8;  // per-thread piece statistics kept in registers

template <int D, int NW>
__global__ void __launch_bounds__(kMergeThreads) attn_tc_merge(const AttnParams p, int32_t ctas) {
    extern __shared__ float fac[];  // [2][pieces][G]: 2^(m - M) per CTA piece and head
    __shared__ float red[kMergeThreads];
    __shared__ float headM[2][16], headInvL[2][16];
    const int32_t c = blockIdx.x;
    __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(p.out);
    // launched as a programmatic dependent of attn_tc_persistent: wait for it,
    // and let the next kernel (the next layer's split) start its prologue
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const TcWs ws = tc_ws(p, ctas, NW, D);
    const CtaHdr Hc = ws.hdr[c];

    if (launch_aborted(p)) return;
    const int64_t P = Hc.P;
    if (P <= 0) return;
    const int G = p.G;

    // the (at most two) cut segments this CTA shares
    int64_t seg0[2];
    int32_t segn[2], segg[2], cf[2], np_[2];
    int nseg = 0;
    for (int which = 0; which < 2; ++which) {
        const int64_t s0 = which == 0 ? Hc.a0 : Hc.b0, s1 = which == 0 ? Hc.a1 : Hc.b1;
        if (s0 < 0 || (which == 1 && s0 == Hc.a0)) continue;
        const int32_t c_first = owner(s0, P, ctas), c_last = owner(s1 - 1, P, ctas);
        // not cut (finished in the split kernel), or this CTA holds none of it
        // (an empty CTA right before c_first starts at the segment's first page)
        if (c_first == c_last || c < c_first || c > c_last) continue;
        seg0[nseg] = s0;
        segn[nseg] = which == 0 ? Hc.an : Hc.bn;
        segg[nseg] = which == 0 ? Hc.ag : Hc.bg;
        cf[nseg] = c_first;
        np_[nseg] = c_last - c_first + 1;
        ++nseg;
    }
    if (nseg == 0) return;
    (void)seg0;
    // threads [0, half) take segment 0, [half, 2 half) segment 1 (all of them
    // take segment 0 when there is only one)
    const int half = nseg == 2 ? kMergeHalf : kMergeThreads;
    const int si = nseg == 2 ? static_cast<int>(threadIdx.x) / kMergeHalf : 0;
    const int tl = static_cast<int>(threadIdx.x) - si * half;  // thread index within the half
    const int32_t c_first = cf[si], np = np_[si];
    const int k = c - c_first;  // this CTA's share of the outputs
    auto nonempty = [&](int32_t cc_) { return P * cc_ / ctas < P * (cc_ + 1) / ctas; };
    // CTA c_first keeps slot 1 (the segment begins in its slice); the others slot 0
    auto piece = [&](int i) -> int64_t {
        return (static_cast<int64_t>(c_first + i) * 2 + (i == 0 ? 1 : 0)) * G;
    };
    float* ftab = fac + si * ctas * G;
    // per-head max and sum over the pieces: thread tl handles head tl % 16
    const int h16 = tl & 15, sub = tl >> 4, nsub = half >> 4;
    float2 mlr[kMergeRegPieces];
    float mloc = -INFINITY;
#pragma unroll
    for (int j = 0; j < kMergeRegPieces; ++j) {
        const int i = sub + j * nsub;
        mlr[j] = make_float2(-INFINITY, 0.f);
        if (h16 < G && i < np && nonempty(c_first + i)) mlr[j] = ws.c_ml[piece(i) + h16];
        mloc = fmaxf(mloc, mlr[j].x);
    }
    for (int i = sub + kMergeRegPieces * nsub; h16 < G && i < np; i += nsub)  // rare: long spans
        if (nonempty(c_first + i)) mloc = fmaxf(mloc, ws.c_ml[piece(i) + h16].x);
    red[threadIdx.x] = mloc;
    __syncthreads();
    if (tl < 16) {
        float M = -INFINITY;
        for (int j = 0; j < nsub; ++j) M = fmaxf(M, red[si * half + j * 16 + tl]);
        headM[si][tl] = M;
    }
    __syncthreads();
    float lloc = 0.f;
    if (h16 < G) {
        const float M = headM[si][h16];
#pragma unroll
        for (int j = 0; j < kMergeRegPieces; ++j) {
            const int i = sub + j * nsub;
            if (i < np) {
                const float f = mlr[j].x != -INFINITY ? exp2_approx(mlr[j].x - M) : 0.f;
                lloc += mlr[j].y * f;
                ftab[i * G + h16] = f;
            }
        }
        for (int i = sub + kMergeRegPieces * nsub; i < np; i += nsub) {
            float f = 0.f;
            if (nonempty(c_first + i)) {
                const float2 ml = ws.c_ml[piece(i) + h16];
                if (ml.x != -INFINITY) f = exp2_approx(ml.x - M);
                lloc += ml.y * f;
            }
            ftab[i * G + h16] = f;
        }
    }
    red[threadIdx.x] = lloc;
    __syncthreads();
    if (tl < 16) {
        float L = 0.f;
        for (int j = 0; j < nsub; ++j) L += red[si * half + j * 16 + tl];
        headInvL[si][tl] = 1.f / L;
    }
    __syncthreads();
    // this CTA's share of the segment's G x D outputs
    const int total = G * D;
    const int per = (total + np - 1) / np;
    const int lo = k * per, hi = min(total, lo + per);
    const int64_t head0 = static_cast<int64_t>(segn[si]) * p.H_q + segg[si] * G;
    const int64_t st = static_cast<int64_t>(2) * G * D;
    for (int idx = lo + tl; idx < hi; idx += half) {
        const int h = idx / D;
        // an empty CTA's slot was never written (stale, maybe NaN): select, never scale by 0
        const float f0 = ftab[h];
        const float v0 = ws.c_o[piece(0) * D + idx];  // slot 1 of c_first
        float acc = f0 != 0.f ? v0 * f0 : 0.f;
        const float* b1 = ws.c_o + (static_cast<int64_t>(c_first) * 2 * G) * D + idx;
        int i = 1;
        for (; i + 8 <= np; i += 8) {  // eight independent loads in flight
            float a[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) a[u] = b1[st * (i + u)];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float f = ftab[(i + u) * G + h];
                acc += f != 0.f ? a[u] * f : 0.f;
            }
        }
        for (; i < np; ++i) {
            const float f = ftab[i * G + h];
            acc += f != 0.f ? b1[st * i] * f : 0.f;
        }
        outp[head0 * D + idx] = __float2bfloat16_rn(acc * headInvL[si][h]);
    }
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

template <int D, int BS, int NT, bool F8>
cudaError_t launch_one(const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p, int sms,
                       cudaStream_t s) {
    using S = TcShape<D, BS, F8, NT>;
    static unsigned long long smem_fwd = 0, smem_rev = 0, smem_fuse = 0;  // one per kernel
    const bool fuse = p.k_new != nullptr;
    auto kernel = fuse ? attn_tc_persistent<D, BS, NT, false, F8, true>
                       : (p.reverse ? attn_tc_persistent<D, BS, NT, true, F8, false>
                                    : attn_tc_persistent<D, BS, NT, false, F8, false>);
    cudaError_t e = ensure_smem_attr(kernel, S::SMEM,
                                     fuse ? smem_fuse : (p.reverse ? smem_rev : smem_fwd));
    if (e != cudaSuccess) return e;
    const int ctas = tc_ctas(sms);
    AttnParams q = p;  // workspace: outputs of all pieces, then their (m, l), then headers
    q.ws_ml = reinterpret_cast<float2*>(p.ws_o + tc_pieces(ctas, S::NW, p.G) * D);
    // The merge grid is a programmatic dependent of the split grid: it is
    // scheduled while the split grid drains and waits (griddepcontrol.wait)
    // before reading its partials. The split grid is one of the kernel before
    // it only when the caller allows the overlap: it then runs its metadata
    // prologue and first page copies while that kernel (for example the
    // previous layer's merge) drains, and waits before it touches queries,
    // outputs or the workspace.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(S::NW * 32);
    cfg.dynamicSmemBytes = S::SMEM;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = p.overlap ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kernel, mk, mv, q);
    if (e != cudaSuccess) return e;
    cfg.numAttrs = 1;
    const int msmem = 2 * ctas * p.G * static_cast<int>(sizeof(float));  // factor tables
    const int msmem_max = 2 * ctas * 16 * static_cast<int>(sizeof(float));  // largest group
    if (msmem_max > 48 * 1024) {  // only ever raise the limit above the default
        static unsigned long long merge_smem_set = 0;
        e = ensure_smem_attr(attn_tc_merge<D, S::NW>, msmem_max, merge_smem_set);
        if (e != cudaSuccess) return e;
    }
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = msmem;
    return cudaLaunchKernelEx(&cfg, attn_tc_merge<D, S::NW>, q, static_cast<int32_t>(ctas));
}

template <int D, bool F8>
cudaError_t launch_d(const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p, int BS,
                     int sms, cudaStream_t s) {
    const bool wide = p.G > 8;
    if (BS == 16) return wide ? launch_one<D, 16, 2, F8>(mk, mv, p, sms, s)
                              : launch_one<D, 16, 1, F8>(mk, mv, p, sms, s);
    return wide ? launch_one<D, 32, 2, F8>(mk, mv, p, sms, s)
                : launch_one<D, 32, 1, F8>(mk, mv, p, sms, s);
}

}  // namespace
}  // namespace yoco
