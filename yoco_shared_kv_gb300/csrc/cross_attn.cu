// yoco_cross_attn_paged: one cross-decoder layer of causal paged GQA attention
// against the single shared K^/V^ cache.
//
// "KV cache memory systems", "Cache contents": out = softmax(q K^T / sqrt(d_h)) V
// over the cached keys up to the query position; the kernel "resolves each
// logical block through the block table" ("Contiguous allocation wastes
// capacity"). "YOCO 论文与推理数据流详解" §10.4 and §11: each of the L/2
// cross-decoder layers sends its own queries against the same shared cache,
// so decode is a stream of the whole cache per layer and is bound by HBM.
//
// Work decomposition (flash-decoding style split-KV):
//   CTA = (cross row n, kv head g, split s). A split is `split_pages`
//   consecutive logical pages of the row's causal range. Inside a CTA each
//   warp owns the pages p = first + warp, first + warp + NW, ... and runs its
//   own online softmax; warps are merged in shared memory, splits by a
//   second kernel with a log-sum-exp combine in split order. Which warp and
//   which split see a page depends only on its logical index, so the result
//   is bit-identical under any physical placement of the pages.
//
// bf16 path (tensor cores): every query head of the kv group shares one read
//   of each K/V page. A page of one kv head is a contiguous [block_size x
//   head_dim] run; TMA copies it into shared memory as head_dim/64 tiles of
//   [block_size x 128 B] with the 128-byte swizzle, so ldmatrix reads are
//   bank-conflict free. S^T = K Q^T and O^T += V^T P^T are m16n8k16 bf16
//   mma.sync products with fp32 accumulators: the group's heads are the N=8
//   (or 16) side, tokens / head dims the M side. P goes from the S^T
//   accumulator layout to the B-operand layout with movmatrix (a register
//   transpose), never through shared memory.
// fp32 path (CUDA cores): one warp per page, lanes across head_dim, warp
//   shuffles for the dot products; exact fp32 arithmetic throughout.
#include <mutex>

#include "common.cuh"

namespace yoco {
namespace {

struct AttnParams {
    const void* q;
    void* out;
    const int32_t* block_table;
    const int32_t* seq_lens;
    const int32_t* cqsl;
    float* ws_o;    // [max_rows][H_q][max_splits][D] unnormalised partial outputs
    float2* ws_ml;  // [max_rows][H_q][max_splits] (running max in log2 units, sum)
    int32_t* err;
    int32_t max_blocks;
    int32_t num_reqs;
    int32_t H_q, H_kv, G;
    int32_t num_blocks;
    int32_t block_size;
    int32_t split_pages;
    int32_t max_splits;
    float scale_log2;  // softmax scale * log2(e)
};

// Wait limit for one asynchronous page copy before the kernel gives up.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Resolve a CTA's row / split. Returns false if the CTA has no work.
// On an empty row the split-0 CTA zero-fills `heads` output heads starting
// at `head0` and flags the error.
template <typename T, int D>
__device__ __forceinline__ bool cta_range(const AttnParams& p, int32_t n, int32_t s, int32_t head0,
                                          int32_t heads, int32_t& req, int32_t& kv_len,
                                          int32_t& p_begin, int32_t& p_end, int32_t& nsplit) {
    if (!locate_row(p.cqsl, p.num_reqs, n, p.seq_lens, req, kv_len)) return false;
    // once some CTA gave up on a copy, the rest of the launch does no work
    if (p.err != nullptr && (*reinterpret_cast<volatile int32_t*>(p.err) & YOCO_DEVERR_TIMEOUT))
        return false;
    if (kv_len <= 0) {
        if (s == 0) {
            T* o = static_cast<T*>(p.out) + (static_cast<int64_t>(n) * p.H_q + head0) * D;
            for (int i = threadIdx.x; i < heads * D; i += blockDim.x) o[i] = T(0.0f);
            if (threadIdx.x == 0) set_err(p.err, YOCO_DEVERR_EMPTY_ROW);
        }
        return false;
    }
    const int64_t cap = static_cast<int64_t>(p.max_blocks) * p.block_size;
    if (kv_len > cap) {
        if (threadIdx.x == 0 && s == 0) set_err(p.err, YOCO_DEVERR_POS_RANGE);
        kv_len = static_cast<int32_t>(cap);
    }
    const int32_t n_pages = (kv_len + p.block_size - 1) / p.block_size;
    nsplit = (n_pages + p.split_pages - 1) / p.split_pages;
    if (s >= nsplit) return false;
    p_begin = s * p.split_pages;
    p_end = min(n_pages, p_begin + p.split_pages);
    return true;
}

template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ float from_float<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Combine per-warp (m, l, o) partials in shared memory and write either the
// final normalised output (single split) or the split's partial.
template <typename T, int D, int NWARP, int NH>
__device__ __forceinline__ void cta_finish(const AttnParams& p, const float* red_m,
                                           const float* red_l, const float* red_o, int32_t n,
                                           int32_t s, int32_t head0, int32_t heads,
                                           int32_t nsplit) {
    for (int idx = threadIdx.x; idx < heads * D; idx += blockDim.x) {
        const int h = idx / D, d = idx - (idx / D) * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NWARP; ++w) M = fmaxf(M, red_m[w * NH + h]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < NWARP; ++w) {
            const float mw = red_m[w * NH + h];
            if (mw == -INFINITY) continue;  // warp saw no page
            const float f = exp2_approx(mw - M);
            L += red_l[w * NH + h] * f;
            O += red_o[(w * NH + h) * D + d] * f;
        }
        const int64_t head = static_cast<int64_t>(n) * p.H_q + head0 + h;
        if (nsplit == 1) {
            static_cast<T*>(p.out)[head * D + d] = from_float<T>(O / L);
        } else {
            const int64_t slot = head * p.max_splits + s;
            p.ws_o[slot * D + d] = O;
            if (d == 0) p.ws_ml[slot] = make_float2(M, L);
        }
    }
}

// ----------------------------------------------------------- bf16 / tensor

template <int D, int BS>
struct TcShape {
    static constexpr int PAGE_BYTES = BS * D * 2;        // K (or V) of one page, one kv head
    static constexpr int STAGE_BYTES = 2 * PAGE_BYTES;   // K + V
    static constexpr int NW = STAGE_BYTES >= 32768 ? 2 : 4;
    static constexpr int STAGES = STAGE_BYTES >= 16384 ? 3 : 4;
    static constexpr int KSUB = D / 64;                  // 128-byte swizzled sub-tiles per row
    static constexpr int SUB_BYTES = BS * 128;
    static constexpr int MT = BS / 16;                   // 16-token tiles per page
    static constexpr int KD = D / 16;                    // 16-wide steps along head_dim
    static constexpr int SMEM = NW * STAGES * STAGE_BYTES + 1024;
};

// Byte offset of (token row t, 16-byte chunk j of head-dim sub-tile c) in a
// 128B-swizzled page tile.
template <int BS>
__device__ __forceinline__ uint32_t swz(int c, int t, int j) {
    return static_cast<uint32_t>(c * (BS * 128) + t * 128 + ((j ^ (t & 7)) << 4));
}

template <int D, int BS, int NT>
__global__ void __launch_bounds__(TcShape<D, BS>::NW * 32, 1)
    attn_split_tc(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const AttnParams p) {
    using S = TcShape<D, BS>;
    constexpr int NW = S::NW, STAGES = S::STAGES, NH = NT * 8;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[NW * STAGES];
    __shared__ int abort_flag;

    const int32_t n = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
    int32_t req, kv_len, p_begin, p_end, nsplit;
    if (!cta_range<__nv_bfloat16, D>(p, n, s, g * p.G, p.G, req, kv_len, p_begin, p_end, nsplit))
        return;

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gl = lane >> 2, tq = lane & 3;  // mma fragment row group / column pair

    if (threadIdx.x == 0) {
        abort_flag = 0;
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    if (lane == 0) {
        for (int i = 0; i < STAGES; ++i) mbar_init(&bars[warp * STAGES + i], 1);
        fence_mbar_init();
    }
    __syncthreads();

    const int32_t* bt_row = p.block_table + static_cast<int64_t>(req) * p.max_blocks;
    const int32_t n_my = (p_end - p_begin - warp + NW - 1) / NW > 0
                             ? (p_end - p_begin - warp + NW - 1) / NW
                             : 0;
    uint8_t* wbuf = smem + warp * STAGES * S::STAGE_BYTES;
    uint64_t* wbar = bars + warp * STAGES;
    const int32_t row0_base = g;  // kv head offset inside a page's rows

    auto issue = [&](int i) {  // lane 0 only
        const int32_t lp = p_begin + warp + i * NW;
        const int st = i % STAGES;
        const int32_t blk = __ldg(bt_row + lp);
        uint64_t* bar = wbar + st;
        if (blk < 0 || blk >= p.num_blocks) {
            set_err(p.err, YOCO_DEVERR_PAGE_RANGE);
            mbar_arrive(bar);
            return;
        }
        mbar_arrive_expect_tx(bar, 2 * S::PAGE_BYTES);
        uint8_t* kd = wbuf + st * S::STAGE_BYTES;
        uint8_t* vd = kd + S::PAGE_BYTES;
        const int32_t y = (blk * p.H_kv + row0_base) * BS;
#pragma unroll
        for (int c = 0; c < S::KSUB; ++c) {
            tma_load_2d(kd + c * S::SUB_BYTES, &tm_k, c * 64, y, bar);
            tma_load_2d(vd + c * S::SUB_BYTES, &tm_v, c * 64, y, bar);
        }
    };

    if (lane == 0) {
        const int pro = n_my < STAGES ? n_my : STAGES;
        for (int i = 0; i < pro; ++i) issue(i);
    }

    // Q fragments (B operand of S^T = K Q^T): head gl of n-tile nt, dims 2tq..
    uint32_t qf[S::KD][NT][2];
    {
        const __nv_bfloat16* qrow =
            static_cast<const __nv_bfloat16*>(p.q) + (static_cast<int64_t>(n) * p.H_q + g * p.G) * D;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int h = nt * 8 + gl;
            const bool ok = h < p.G;
            const uint32_t* src = reinterpret_cast<const uint32_t*>(qrow + (ok ? h : 0) * D);
#pragma unroll
            for (int kk = 0; kk < S::KD; ++kk) {
                qf[kk][nt][0] = ok ? __ldg(src + (kk * 16 + 2 * tq) / 2) : 0u;
                qf[kk][nt][1] = ok ? __ldg(src + (kk * 16 + 8 + 2 * tq) / 2) : 0u;
            }
        }
    }

    float o[S::KD][NT][4];
#pragma unroll
    for (int a = 0; a < S::KD; ++a)
#pragma unroll
        for (int b = 0; b < NT; ++b)
#pragma unroll
            for (int c = 0; c < 4; ++c) o[a][b][c] = 0.f;
    float m_run[NT][2], l_part[NT][2];
#pragma unroll
    for (int b = 0; b < NT; ++b) {
        m_run[b][0] = m_run[b][1] = -INFINITY;
        l_part[b][0] = l_part[b][1] = 0.f;
    }
    const float sl2 = p.scale_log2;
    bool aborted = false;
    int consumed = 0;

    for (int i = 0; i < n_my; ++i) {
        const int st = i % STAGES;
        if (!mbar_wait_bounded(wbar + st, (i / STAGES) & 1, kWaitLimitNs)) {
            aborted = true;
            break;
        }
        consumed = i + 1;
        const int32_t lp = p_begin + warp + i * NW;
        const int32_t blk = __ldg(bt_row + lp);
        if (blk >= 0 && blk < p.num_blocks) {
            const uint32_t kbase = smem_u32(wbuf + st * S::STAGE_BYTES);
            const uint32_t vbase = kbase + S::PAGE_BYTES;
            const int32_t nvalid = min(BS, kv_len - lp * BS);
            if (nvalid < BS) {
                // Rows past the causal end may hold stale data (even NaN); a
                // zero probability times NaN is NaN, so clear those V rows.
                uint8_t* vd = wbuf + st * S::STAGE_BYTES + S::PAGE_BYTES;
                const int nbytes = (BS - nvalid) * 128;
                for (int c = 0; c < S::KSUB; ++c)
                    for (int b = lane * 16; b < nbytes; b += 32 * 16)
                        *reinterpret_cast<uint4*>(vd + c * S::SUB_BYTES + nvalid * 128 + b) =
                            make_uint4(0, 0, 0, 0);
                fence_proxy_async_smem();
                __syncwarp();
            }
            // ---- S^T = K Q^T  (tokens x heads) ----
            float sc[S::MT][NT][4];
#pragma unroll
            for (int mt = 0; mt < S::MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int c = 0; c < 4; ++c) sc[mt][nt][c] = 0.f;
            {
                const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
                for (int mt = 0; mt < S::MT; ++mt) {
                    const int t = mt * 16 + (mi & 1) * 8 + rr;
#pragma unroll
                    for (int kk = 0; kk < S::KD; ++kk) {
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4(kbase + swz<BS>(kk >> 2, t, (kk & 3) * 2 + (mi >> 1)), a0, a1, a2,
                                a3);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma_bf16_16816(sc[mt][nt], a0, a1, a2, a3, qf[kk][nt][0],
                                           qf[kk][nt][1]);
                    }
                }
            }
            // ---- online softmax (log2 domain) ----
            float corr[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int mt = 0; mt < S::MT; ++mt) {
                    const int t0 = mt * 16 + gl, t1 = t0 + 8;
                    float* c = sc[mt][nt];
                    c[0] = t0 < nvalid ? c[0] * sl2 : -INFINITY;
                    c[1] = t0 < nvalid ? c[1] * sl2 : -INFINITY;
                    c[2] = t1 < nvalid ? c[2] * sl2 : -INFINITY;
                    c[3] = t1 < nvalid ? c[3] * sl2 : -INFINITY;
                    mx0 = fmaxf(mx0, fmaxf(c[0], c[2]));
                    mx1 = fmaxf(mx1, fmaxf(c[1], c[3]));
                }
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                }
                const float mn0 = fmaxf(m_run[nt][0], mx0), mn1 = fmaxf(m_run[nt][1], mx1);
                corr[nt][0] = exp2_approx(m_run[nt][0] - mn0);
                corr[nt][1] = exp2_approx(m_run[nt][1] - mn1);
                m_run[nt][0] = mn0;
                m_run[nt][1] = mn1;
            }
            // rescale the running output where the max moved
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
#pragma unroll
            for (int kt = 0; kt < S::MT; ++kt) {
                uint32_t pb[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float* c = sc[kt][nt];
                    const uint32_t lo = pack_bf16x2(exp2_approx(c[0] - m_run[nt][0]),
                                                    exp2_approx(c[1] - m_run[nt][1]));
                    const uint32_t hi = pack_bf16x2(exp2_approx(c[2] - m_run[nt][0]),
                                                    exp2_approx(c[3] - m_run[nt][1]));
                    // the row sums use exactly the rounded weights fed to the mma
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
                    ldsm_x4_trans(vbase + swz<BS>(md >> 2, t, (md & 3) * 2 + (mi & 1)), a0, a1, a2,
                                  a3);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_bf16_16816(o[md][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
                }
            }
        }
        __syncwarp();
        if (lane == 0 && i + STAGES < n_my) issue(i + STAGES);
    }

    if (aborted) {
        // Drain copies this warp still has in flight before the CTA exits.
        const int issued = n_my < consumed + STAGES ? n_my : consumed + STAGES;
        for (int i = consumed; i < issued; ++i)
            (void)mbar_wait_bounded(wbar + (i % STAGES), (i / STAGES) & 1, kWaitLimitNs);
        if (lane == 0) {
            set_err(p.err, YOCO_DEVERR_TIMEOUT);
            atomicExch(&abort_flag, 1);
        }
    }

    // row sums: reduce the per-thread partials over the 8 row groups
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l_part[nt][0] += __shfl_xor_sync(0xffffffffu, l_part[nt][0], off);
            l_part[nt][1] += __shfl_xor_sync(0xffffffffu, l_part[nt][1], off);
        }

    __syncthreads();  // every warp is done with its stages: reuse them
    float* red_m = reinterpret_cast<float*>(smem);
    float* red_l = red_m + NW * NH;
    float* red_o = red_l + NW * NH;  // [NW][NH][D]
    if (gl == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            red_m[warp * NH + nt * 8 + 2 * tq] = m_run[nt][0];
            red_m[warp * NH + nt * 8 + 2 * tq + 1] = m_run[nt][1];
            red_l[warp * NH + nt * 8 + 2 * tq] = l_part[nt][0];
            red_l[warp * NH + nt * 8 + 2 * tq + 1] = l_part[nt][1];
        }
    }
#pragma unroll
    for (int md = 0; md < S::KD; ++md)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int h0 = nt * 8 + 2 * tq, d0 = md * 16 + gl;
            float* base = red_o + static_cast<size_t>(warp * NH) * D;
            base[h0 * D + d0] = o[md][nt][0];
            base[(h0 + 1) * D + d0] = o[md][nt][1];
            base[h0 * D + d0 + 8] = o[md][nt][2];
            base[(h0 + 1) * D + d0 + 8] = o[md][nt][3];
        }
    __syncthreads();
    if (abort_flag) return;
    cta_finish<__nv_bfloat16, D, NW, NH>(p, red_m, red_l, red_o, n, s, g * p.G, p.G, nsplit);
}

// -------------------------------------------------------------- fp32 / CUDA cores

constexpr int kCcWarps = 4;

template <typename T>
__device__ __forceinline__ float load_f(const T* p);
template <>
__device__ __forceinline__ float load_f<float>(const float* p) { return __ldg(p); }

template <typename T, int D, int HB>
__global__ void __launch_bounds__(kCcWarps * 32)
    attn_split_cc(const T* __restrict__ k_cache, const T* __restrict__ v_cache, const AttnParams p) {
    constexpr int E = D / 32;
    __shared__ float red_m[kCcWarps * HB], red_l[kCcWarps * HB];
    __shared__ float red_o[kCcWarps * HB * D];

    const int32_t n = blockIdx.x, hc = blockIdx.y, s = blockIdx.z;
    const int32_t head0 = hc * HB, g = head0 / p.G;
    int32_t req, kv_len, p_begin, p_end, nsplit;
    if (!cta_range<T, D>(p, n, s, head0, HB, req, kv_len, p_begin, p_end, nsplit)) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const T* qrow = static_cast<const T*>(p.q) + (static_cast<int64_t>(n) * p.H_q + head0) * D;
    float qv[HB][E], o[HB][E], m[HB], l[HB];
#pragma unroll
    for (int h = 0; h < HB; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            qv[h][e] = load_f<T>(qrow + h * D + lane + 32 * e) * p.scale_log2;
            o[h][e] = 0.f;
        }
    }
    const int32_t* bt_row = p.block_table + static_cast<int64_t>(req) * p.max_blocks;
    const int bs = p.block_size;
    for (int32_t lp = p_begin + warp; lp < p_end; lp += kCcWarps) {
        const int32_t blk = __ldg(bt_row + lp);
        if (blk < 0 || blk >= p.num_blocks) {
            if (lane == 0) set_err(p.err, YOCO_DEVERR_PAGE_RANGE);
            continue;
        }
        const int ntok = min(bs, kv_len - lp * bs);
        const int64_t base = (static_cast<int64_t>(blk) * p.H_kv + g) * bs * D;
        for (int tt = 0; tt < ntok; ++tt) {
            float kk[E], vv[E];
#pragma unroll
            for (int e = 0; e < E; ++e) {
                kk[e] = load_f<T>(k_cache + base + tt * D + lane + 32 * e);
                vv[e] = load_f<T>(v_cache + base + tt * D + lane + 32 * e);
            }
#pragma unroll
            for (int h = 0; h < HB; ++h) {
                float sdot = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) sdot = fmaf(qv[h][e], kk[e], sdot);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    sdot += __shfl_xor_sync(0xffffffffu, sdot, off);
                const float mn = fmaxf(m[h], sdot);
                const float corr = exp2_approx(m[h] - mn);
                const float pe = exp2_approx(sdot - mn);
                l[h] = l[h] * corr + pe;
#pragma unroll
                for (int e = 0; e < E; ++e) o[h][e] = fmaf(o[h][e], corr, pe * vv[e]);
                m[h] = mn;
            }
        }
    }
#pragma unroll
    for (int h = 0; h < HB; ++h) {
        if (lane == 0) {
            red_m[warp * HB + h] = m[h];
            red_l[warp * HB + h] = l[h];
        }
#pragma unroll
        for (int e = 0; e < E; ++e) red_o[(warp * HB + h) * D + lane + 32 * e] = o[h][e];
    }
    __syncthreads();
    cta_finish<T, D, kCcWarps, HB>(p, red_m, red_l, red_o, n, s, head0, HB, nsplit);
}

// ------------------------------------------------------------ split merge

constexpr int kMergeThreads = 128;

template <typename T, int D>
__global__ void __launch_bounds__(kMergeThreads) attn_merge(const AttnParams p) {
    const int32_t n = blockIdx.x, h = blockIdx.y;
    int32_t req, kv_len;
    if (!locate_row(p.cqsl, p.num_reqs, n, p.seq_lens, req, kv_len) || kv_len <= 0) return;
    const int64_t cap = static_cast<int64_t>(p.max_blocks) * p.block_size;
    if (kv_len > cap) kv_len = static_cast<int32_t>(cap);
    const int32_t n_pages = (kv_len + p.block_size - 1) / p.block_size;
    const int32_t nsplit = (n_pages + p.split_pages - 1) / p.split_pages;
    if (nsplit <= 1) return;
    const int64_t head = static_cast<int64_t>(n) * p.H_q + h;
    const float2* ml = p.ws_ml + head * p.max_splits;
    float M = -INFINITY;
    for (int32_t s = 0; s < nsplit; ++s) M = fmaxf(M, ml[s].x);
    float L = 0.f;
    for (int32_t s = 0; s < nsplit; ++s) L += ml[s].y * exp2_approx(ml[s].x - M);
    const float invL = 1.f / L;
    const float* wo = p.ws_o + head * p.max_splits * D;
    for (int d = threadIdx.x; d < D; d += kMergeThreads) {
        float acc = 0.f;
        for (int32_t s = 0; s < nsplit; ++s) acc += wo[s * D + d] * exp2_approx(ml[s].x - M);
        static_cast<T*>(p.out)[head * D + d] = from_float<T>(acc * invL);
    }
}

// ------------------------------------------------------------------- host

struct Plan {
    bool tc;          // tensor-core bf16 path
    int nw;           // warps per CTA (pages round-robin over them)
    int hb;           // CUDA-core path: query heads per CTA
    int split_pages;  // logical pages per split
    int max_splits;
    size_t ws_bytes;
};

int tc_warps(int D, int BS) {
    switch (D * 100 + BS) {  // must match TcShape<D, BS>::NW
        case 6416: return TcShape<64, 16>::NW;
        case 6432: return TcShape<64, 32>::NW;
        case 12816: return TcShape<128, 16>::NW;
        case 12832: return TcShape<128, 32>::NW;
        case 25616: return TcShape<256, 16>::NW;
        default: return TcShape<256, 32>::NW;
    }
}

bool make_plan(yoco_dtype_t dt, int max_rows, int H_q, int H_kv, int D, int BS, int max_seq_len,
               Plan& pl) {
    if (!dtype_ok(dt) || !head_dim_ok(D) || !block_size_ok(BS)) return false;
    if (H_q <= 0 || H_kv <= 0 || H_q % H_kv != 0 || H_q / H_kv > 16) return false;
    if (max_rows < 0 || max_seq_len <= 0) return false;
    const int G = H_q / H_kv;
    pl.tc = (dt == YOCO_BF16);
    pl.hb = 1;
    int units;
    if (pl.tc) {
        pl.nw = tc_warps(D, BS);
        units = H_kv;
    } else {
        pl.nw = kCcWarps;
        for (int c : {8, 4, 2, 1})
            if (G % c == 0) {
                pl.hb = c;
                break;
            }
        units = H_q / pl.hb;
    }
    const int64_t pages_max = (static_cast<int64_t>(max_seq_len) + BS - 1) / BS;
    const int64_t target = 8ll * device_sm_count();  // CTAs to aim for at the bound
    const int64_t unit_total = static_cast<int64_t>(max_rows > 0 ? max_rows : 1) * units;
    const int64_t want = (target + unit_total - 1) / unit_total;
    int64_t sp = (pages_max + want - 1) / want;
    const int64_t min_pages = static_cast<int64_t>(pl.nw) * 8;
    if (sp < min_pages) sp = min_pages;
    sp = (sp + pl.nw - 1) / pl.nw * pl.nw;
    if (sp > (1ll << 30)) return false;
    pl.split_pages = static_cast<int>(sp);
    pl.max_splits = static_cast<int>((pages_max + sp - 1) / sp);
    if (pl.max_splits > 65535) return false;
    pl.ws_bytes = pl.max_splits > 1
                      ? static_cast<size_t>(max_rows) * H_q * pl.max_splits *
                            (static_cast<size_t>(D) * 4 + 8)
                      : 0;
    return true;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// Pool [num_blocks * H_kv * BS rows][D] bf16 as a 2-D tensor; box = 64 elements
// (128 bytes) x BS rows, 128-byte swizzle.
bool encode_pool(CUtensorMap* map, const void* pool, int64_t rows, int D, int BS) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(BS)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int BS, int NT>
cudaError_t launch_tc(const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p,
                      dim3 grid, cudaStream_t s) {
    using S = TcShape<D, BS>;
    cudaError_t e = cudaFuncSetAttribute(attn_split_tc<D, BS, NT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
    if (e != cudaSuccess) return e;
    attn_split_tc<D, BS, NT><<<grid, S::NW * 32, S::SMEM, s>>>(mk, mv, p);
    return cudaGetLastError();
}

template <int D>
cudaError_t dispatch_tc(int BS, int NT, const CUtensorMap& mk, const CUtensorMap& mv,
                        const AttnParams& p, dim3 grid, cudaStream_t s) {
    if (BS == 16) return NT == 1 ? launch_tc<D, 16, 1>(mk, mv, p, grid, s)
                                 : launch_tc<D, 16, 2>(mk, mv, p, grid, s);
    return NT == 1 ? launch_tc<D, 32, 1>(mk, mv, p, grid, s) : launch_tc<D, 32, 2>(mk, mv, p, grid, s);
}

template <typename T, int D>
cudaError_t dispatch_cc(int hb, const void* kc, const void* vc, const AttnParams& p, dim3 grid,
                        cudaStream_t s) {
    const T* k = static_cast<const T*>(kc);
    const T* v = static_cast<const T*>(vc);
    switch (hb) {
        case 8: attn_split_cc<T, D, 8><<<grid, kCcWarps * 32, 0, s>>>(k, v, p); break;
        case 4: attn_split_cc<T, D, 4><<<grid, kCcWarps * 32, 0, s>>>(k, v, p); break;
        case 2: attn_split_cc<T, D, 2><<<grid, kCcWarps * 32, 0, s>>>(k, v, p); break;
        default: attn_split_cc<T, D, 1><<<grid, kCcWarps * 32, 0, s>>>(k, v, p); break;
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_merge(int D, const AttnParams& p, dim3 grid, cudaStream_t s) {
    switch (D) {
        case 64: attn_merge<T, 64><<<grid, kMergeThreads, 0, s>>>(p); break;
        case 128: attn_merge<T, 128><<<grid, kMergeThreads, 0, s>>>(p); break;
        default: attn_merge<T, 256><<<grid, kMergeThreads, 0, s>>>(p); break;
    }
    return cudaGetLastError();
}

}  // namespace

int device_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return 148;
    return sms;
}

}  // namespace yoco

extern "C" size_t yoco_cross_attn_workspace_size(int32_t max_rows, int32_t num_q_heads,
                                                 int32_t num_kv_heads, int32_t head_dim,
                                                 int32_t block_size, int32_t max_seq_len,
                                                 yoco_dtype_t dtype) {
    yoco::Plan pl;
    if (!yoco::make_plan(dtype, max_rows, num_q_heads, num_kv_heads, head_dim, block_size,
                         max_seq_len, pl))
        return 0;
    return pl.ws_bytes;
}

extern "C" yoco_status_t yoco_cross_attn_paged(
    const void* q, const void* k_cache, const void* v_cache, void* out, const int32_t* block_table,
    int32_t max_blocks_per_req, const int32_t* seq_lens, const int32_t* cross_query_start_loc,
    int32_t num_reqs, int32_t max_rows, int32_t max_seq_len, int32_t num_q_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale,
    yoco_dtype_t dtype, void* workspace, size_t workspace_bytes, int32_t* err_word, void* stream) {
    using namespace yoco;
    if (!dtype_ok(dtype) || !head_dim_ok(head_dim) || !block_size_ok(block_size))
        return YOCO_ERR_UNSUPPORTED;
    if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return YOCO_ERR_INVALID_ARG;
    if (num_q_heads / num_kv_heads > 16) return YOCO_ERR_UNSUPPORTED;
    if (num_reqs < 0 || max_rows < 0 || max_seq_len <= 0 || num_blocks <= 0 ||
        max_blocks_per_req <= 0 || !(scale > 0.f) || max_rows > 0x7fffffff / num_q_heads)
        return YOCO_ERR_INVALID_ARG;
    if (num_reqs == 0 || max_rows == 0) return YOCO_OK;
    if (!q || !k_cache || !v_cache || !out || !block_table || !seq_lens || !cross_query_start_loc)
        return YOCO_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        (workspace && !aligned16(workspace)))
        return YOCO_ERR_INVALID_ARG;
    // TMA row coordinates are signed 32-bit
    if (static_cast<int64_t>(num_blocks) * num_kv_heads * block_size > 0x7fffffffll)
        return YOCO_ERR_UNSUPPORTED;
    Plan pl;
    if (!make_plan(dtype, max_rows, num_q_heads, num_kv_heads, head_dim, block_size, max_seq_len,
                   pl))
        return YOCO_ERR_UNSUPPORTED;
    if (pl.ws_bytes > 0 && (workspace == nullptr || workspace_bytes < pl.ws_bytes))
        return YOCO_ERR_WORKSPACE;

    AttnParams p;
    p.q = q;
    p.out = out;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.cqsl = cross_query_start_loc;
    p.ws_o = static_cast<float*>(workspace);
    p.ws_ml = reinterpret_cast<float2*>(
        static_cast<uint8_t*>(workspace) +
        static_cast<size_t>(max_rows) * num_q_heads * pl.max_splits * head_dim * 4);
    p.err = err_word;
    p.max_blocks = max_blocks_per_req;
    p.num_reqs = num_reqs;
    p.H_q = num_q_heads;
    p.H_kv = num_kv_heads;
    p.G = num_q_heads / num_kv_heads;
    p.num_blocks = num_blocks;
    p.block_size = block_size;
    p.split_pages = pl.split_pages;
    p.max_splits = pl.max_splits;
    p.scale_log2 = scale * kLog2e;
    if (pl.max_splits <= 1) {
        p.ws_o = nullptr;
        p.ws_ml = nullptr;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (pl.tc) {
        CUtensorMap mk, mv;
        const int64_t rows = static_cast<int64_t>(num_blocks) * num_kv_heads * block_size;
        if (!encode_pool(&mk, k_cache, rows, head_dim, block_size) ||
            !encode_pool(&mv, v_cache, rows, head_dim, block_size))
            return YOCO_ERR_CUDA;
        const dim3 grid(max_rows, num_kv_heads, pl.max_splits);
        const int NT = p.G > 8 ? 2 : 1;
        switch (head_dim) {
            case 64: e = dispatch_tc<64>(block_size, NT, mk, mv, p, grid, s); break;
            case 128: e = dispatch_tc<128>(block_size, NT, mk, mv, p, grid, s); break;
            default: e = dispatch_tc<256>(block_size, NT, mk, mv, p, grid, s); break;
        }
    } else {
        const dim3 grid(max_rows, num_q_heads / pl.hb, pl.max_splits);
        switch (head_dim) {
            case 64: e = dispatch_cc<float, 64>(pl.hb, k_cache, v_cache, p, grid, s); break;
            case 128: e = dispatch_cc<float, 128>(pl.hb, k_cache, v_cache, p, grid, s); break;
            default: e = dispatch_cc<float, 256>(pl.hb, k_cache, v_cache, p, grid, s); break;
        }
    }
    if (e != cudaSuccess) return YOCO_ERR_CUDA;
    if (pl.max_splits > 1) {
        const dim3 mgrid(max_rows, num_q_heads);
        e = dtype == YOCO_BF16 ? dispatch_merge<__nv_bfloat16>(head_dim, p, mgrid, s)
                               : dispatch_merge<float>(head_dim, p, mgrid, s);
        if (e != cudaSuccess) return YOCO_ERR_CUDA;
    }
    return YOCO_OK;
}
