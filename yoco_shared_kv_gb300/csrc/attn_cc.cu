// CUDA-core (fp32) cross-decoder attention: flash-decoding with split-KV.
//
// "KV cache memory systems", "Cache contents": out = softmax(q K^T/sqrt(d_h)) V
// over the cached keys, each logical block resolved through the block table.
// Grid: (cross row, group of query heads, split of the row's pages); four
// warps per CTA take the split's pages round robin, one token at a time with
// lanes across head_dim and warp shuffles for the dot products, each warp
// with its own online softmax. Warps are combined in shared memory and
// splits by attn_merge_cc with a log-sum-exp combine in split order.
// Everything is exact fp32 arithmetic (exp2 in the log2 domain).
#include "attn_common.cuh"

namespace yoco {
namespace {

// Keys a row may attend on this path: the block table's reach and the
// caller's max_seq_len, whichever is smaller.
__device__ __forceinline__ int32_t row_key_cap(const AttnParams& p) {
    const int64_t bt = static_cast<int64_t>(p.max_blocks) * p.block_size;
    return static_cast<int32_t>(bt < p.max_seq_len ? bt : p.max_seq_len);
}

// Resolve a CTA's row / split. Returns false if the CTA has no work.
// On an empty row the split-0 CTA zero-fills `heads` output heads starting
// at `head0` and flags the error.
template <typename T, int D>
__device__ __forceinline__ bool cta_range(const AttnParams& p, int32_t n, int32_t s, int32_t head0,
                                          int32_t heads, int32_t& req, int32_t& kv_len,
                                          int32_t& p_begin, int32_t& p_end, int32_t& nsplit) {
    if (!locate_row(p.cqsl, p.num_reqs, n, p.seq_lens, req, kv_len)) return false;
    if (kv_len <= 0) {
        if (s == 0) {
            T* o = static_cast<T*>(p.out) + (static_cast<int64_t>(n) * p.H_q + head0) * D;
            for (int i = threadIdx.x; i < heads * D; i += blockDim.x) o[i] = T(0.0f);
            if (threadIdx.x == 0) set_err(p.err, YOCO_DEVERR_EMPTY_ROW);
        }
        return false;
    }
    // The split plan (and the workspace) hold max_seq_len keys per row: a row
    // with more (seq_lens above the caller's bound) is cut to that many and
    // flagged, so that no split slot past max_splits is ever written or read.
    const int32_t cap = row_key_cap(p);
    if (kv_len > cap) {
        if (threadIdx.x == 0 && s == 0) set_err(p.err, YOCO_DEVERR_POS_RANGE);
        kv_len = cap;
    }
    const int32_t n_pages = (kv_len + p.block_size - 1) / p.block_size;
    nsplit = (n_pages + p.split_pages - 1) / p.split_pages;
    if (nsplit > p.max_splits) nsplit = p.max_splits;  // unreachable after the cut; kept as a bound
    if (s >= nsplit) return false;
    p_begin = s * p.split_pages;
    p_end = min(n_pages, p_begin + p.split_pages);
    return true;
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

constexpr int kMergeThreads = 128;

template <typename T, int D>
__global__ void __launch_bounds__(kMergeThreads) attn_merge_cc(const AttnParams p) {
    const int32_t n = blockIdx.x, h = blockIdx.y;
    int32_t req, kv_len;
    if (!locate_row(p.cqsl, p.num_reqs, n, p.seq_lens, req, kv_len) || kv_len <= 0) return;
    const int32_t cap = row_key_cap(p);  // the same cut as the split kernel's
    if (kv_len > cap) kv_len = cap;
    const int32_t n_pages = (kv_len + p.block_size - 1) / p.block_size;
    int32_t nsplit = (n_pages + p.split_pages - 1) / p.split_pages;
    if (nsplit > p.max_splits) nsplit = p.max_splits;
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


template <int D>
cudaError_t launch_d(int hb, const void* kc, const void* vc, const AttnParams& p, dim3 grid,
                     cudaStream_t s) {
    const float* k = static_cast<const float*>(kc);
    const float* v = static_cast<const float*>(vc);
    switch (hb) {
        case 8: attn_split_cc<float, D, 8><<<grid, kCcWarps * 32, 0, s>>>(k, v, p); break;
        case 4: attn_split_cc<float, D, 4><<<grid, kCcWarps * 32, 0, s>>>(k, v, p); break;
        case 2: attn_split_cc<float, D, 2><<<grid, kCcWarps * 32, 0, s>>>(k, v, p); break;
        default: attn_split_cc<float, D, 1><<<grid, kCcWarps * 32, 0, s>>>(k, v, p); break;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || p.max_splits <= 1) return e;
    attn_merge_cc<float, D><<<dim3(p.max_rows, p.H_q), kMergeThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_cc(const void* k_cache, const void* v_cache, const AttnParams& p, int D,
                           int hb, cudaStream_t s) {
    const dim3 grid(p.max_rows, p.H_q / hb, p.max_splits);
    switch (D) {
        case 64: return launch_d<64>(hb, k_cache, v_cache, p, grid, s);
        case 128: return launch_d<128>(hb, k_cache, v_cache, p, grid, s);
        default: return launch_d<256>(hb, k_cache, v_cache, p, grid, s);
    }
}

}  // namespace yoco
