// yoco_kv_append: write a step's new shared K^/V^ rows into the paged cache.
//
// "YOCO 论文与推理数据流详解" §7.3 and §10.3: each token's K^/V^ is produced
// once at the self-decoder boundary and appended once to the one global
// cache. "KV cache memory systems", "Contiguous allocation wastes capacity":
// a token's logical block resolves to a physical page through the block table.
//
// The e4m3 variant ("KV cache memory systems", "Quantized cache changes
// attention inputs") stores each element as an 8-bit code of value / scale,
// with a K and a V scale per (page, kv head).
//
// Design: one warp per token copies the token's rows of K and of V for every
// kv head, 16 bytes per lane per instruction. The request of a token is found
// once by a binary search over query_start_loc (no host-side slot_mapping, so
// the call is graph-capturable); index arithmetic stays in shifts and masks
// (block_size 16 or 32), so the copy, not the bookkeeping, bounds the kernel.
#include "common.cuh"

namespace yoco {
namespace {

constexpr int kAppendWarps = 8;

// Request, position and physical page of token tok, with the error checks of
// the append (shared by both caches). Returns false (after setting the error
// bit) when the token must be skipped.
__device__ __forceinline__ bool locate_token(int32_t tok, const int32_t* __restrict__ qsl,
                                             int32_t num_reqs, int32_t last,
                                             const int32_t* __restrict__ seq_lens,
                                             const int32_t* __restrict__ block_table,
                                             int32_t max_blocks, int32_t num_blocks,
                                             int32_t bshift, int lane, int32_t* err,
                                             int64_t& pos, int32_t& page) {
    if (tok >= last || __ldg(qsl) > tok) {  // token outside every request's range
        if (lane == 0) set_err(err, YOCO_DEVERR_OFFSETS);
        return false;
    }
    // first r with qsl[r + 1] > tok
    int32_t lo = 0, hi = num_reqs - 1;
    while (lo < hi) {
        const int32_t mid = (lo + hi) >> 1;
        if (__ldg(qsl + mid + 1) > tok) hi = mid;
        else lo = mid + 1;
    }
    const int32_t q0 = __ldg(qsl + lo), q1 = __ldg(qsl + lo + 1);
    const int32_t q_len = q1 - q0;
    pos = static_cast<int64_t>(__ldg(seq_lens + lo)) - q_len + (tok - q0);
    if (q_len <= 0) {
        if (lane == 0) set_err(err, YOCO_DEVERR_OFFSETS);
        return false;
    }
    if (pos < 0 || (pos >> bshift) >= max_blocks) {
        if (lane == 0) set_err(err, YOCO_DEVERR_POS_RANGE);
        return false;
    }
    page = __ldg(block_table + static_cast<int64_t>(lo) * max_blocks + (pos >> bshift));
    if (page < 0 || page >= num_blocks) {
        if (lane == 0) set_err(err, YOCO_DEVERR_PAGE_RANGE);
        return false;
    }
    return true;
}

// One warp per token: the token's request, position and page are found once
// and its H_kv rows of K and of V (contiguous in k_new / v_new) are copied
// with the lanes striding over all of them, four 16-byte vectors of K and of
// V in flight per lane before the stores.
template <int ROW_VECS>  // 16-byte vectors per (token, head) row
__global__ void __launch_bounds__(kAppendWarps * 32)
    kv_append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                     uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                     const int32_t* __restrict__ block_table, int32_t max_blocks,
                     const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ qsl,
                     int32_t num_reqs, int32_t num_tokens, int32_t num_blocks, int32_t block_size,
                     int32_t num_kv_heads, int32_t* err) {
    constexpr int RSH = ROW_VECS == 8 ? 3 : ROW_VECS == 16 ? 4 : ROW_VECS == 32 ? 5 : 6;
    static_assert((1 << RSH) == ROW_VECS, "rows of 8, 16, 32 or 64 vectors");
    constexpr int U = 4;
    const int lane = threadIdx.x & 31;
    const int32_t warp0 = static_cast<int32_t>(blockIdx.x) * kAppendWarps + (threadIdx.x >> 5);
    const int32_t wstride = static_cast<int32_t>(gridDim.x) * kAppendWarps;
    const int32_t last = __ldg(qsl + num_reqs);
    const int32_t bshift = block_size == 16 ? 4 : 5;
    const int32_t nvec = num_kv_heads * ROW_VECS;  // vectors of one token (all heads)
    for (int32_t tok = warp0; tok < num_tokens; tok += wstride) {
        int64_t pos;
        int32_t page;
        if (!locate_token(tok, qsl, num_reqs, last, seq_lens, block_table, max_blocks, num_blocks,
                          bshift, lane, err, pos, page))
            continue;
        // vector v of the token: head v >> RSH, vector v & (ROW_VECS - 1) of its row
        const int64_t dst0 = (static_cast<int64_t>(page) * num_kv_heads * block_size +
                              (pos & (block_size - 1))) * ROW_VECS;
        const int64_t hstride = static_cast<int64_t>(block_size) * ROW_VECS;
        const uint4* ks = k_new + static_cast<int64_t>(tok) * nvec;
        const uint4* vs = v_new + static_cast<int64_t>(tok) * nvec;
        for (int32_t v0 = lane; v0 < nvec; v0 += 32 * U) {
            uint4 kr[U], vr[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int32_t v = v0 + u * 32;
                if (v < nvec) {
                    kr[u] = __ldcs(ks + v);  // read once: stream past L1/L2
                    vr[u] = __ldcs(vs + v);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int32_t v = v0 + u * 32;
                if (v < nvec) {
                    const int64_t d = dst0 + (v >> RSH) * hstride + (v & (ROW_VECS - 1));
                    k_cache[d] = kr[u];
                    v_cache[d] = vr[u];
                }
            }
        }
    }
}

template <int ROW_VECS>
cudaError_t launch_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                          const int32_t* bt, int32_t max_blocks, const int32_t* seq_lens,
                          const int32_t* qsl, int32_t num_reqs, int32_t num_tokens,
                          int32_t num_blocks, int32_t bs, int32_t H_kv, int32_t* err,
                          cudaStream_t s) {
    int64_t blocks = (static_cast<int64_t>(num_tokens) + kAppendWarps - 1) / kAppendWarps;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    kv_append_kernel<ROW_VECS><<<static_cast<unsigned>(blocks), kAppendWarps * 32, 0, s>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), bt, max_blocks, seq_lens, qsl,
        num_reqs, num_tokens, num_blocks, bs, H_kv, err);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- e4m3 cache

// Same token walk as kv_append_kernel; for each kv head, each lane quantises
// D / 32 consecutive elements of K and of V (value / scale in float32, then
// the nearest code).
template <int D>
__global__ void __launch_bounds__(kAppendWarps * 32)
    kv_append_e4m3_kernel(const __nv_bfloat16* __restrict__ k_new,
                          const __nv_bfloat16* __restrict__ v_new, uint8_t* __restrict__ k_cache,
                          uint8_t* __restrict__ v_cache, const float4* __restrict__ scales,
                          const int32_t* __restrict__ block_table, int32_t max_blocks,
                          const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ qsl,
                          int32_t num_reqs, int32_t num_tokens, int32_t num_blocks,
                          int32_t block_size, int32_t num_kv_heads, int32_t* err) {
    constexpr int E = D / 32;  // elements per lane: 4 or 8
    static_assert(E == 4 || E == 8, "head_dim 128 or 256");
    const int lane = threadIdx.x & 31;
    const int32_t warp0 = static_cast<int32_t>(blockIdx.x) * kAppendWarps + (threadIdx.x >> 5);
    const int32_t wstride = static_cast<int32_t>(gridDim.x) * kAppendWarps;
    const int32_t last = __ldg(qsl + num_reqs);
    const int32_t bshift = block_size == 16 ? 4 : 5;
    for (int32_t tok = warp0; tok < num_tokens; tok += wstride) {
        int64_t pos;
        int32_t page;
        if (!locate_token(tok, qsl, num_reqs, last, seq_lens, block_table, max_blocks, num_blocks,
                          bshift, lane, err, pos, page))
            continue;
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            const float4 sc = __ldg(scales + static_cast<int64_t>(page) * num_kv_heads + h);
            if (!scale_usable(sc.x) || !scale_usable(sc.y)) {
                if (lane == 0) set_err(err, YOCO_DEVERR_SCALE);
                continue;
            }
            const int64_t dst = ((static_cast<int64_t>(page) * num_kv_heads + h) * block_size +
                                 (pos & (block_size - 1))) * D + lane * E;
            const int64_t src = (static_cast<int64_t>(tok) * num_kv_heads + h) * D + lane * E;
            if constexpr (E == 4) {
                const uint2 kb = __ldcs(reinterpret_cast<const uint2*>(k_new + src));
                const uint2 vb = __ldcs(reinterpret_cast<const uint2*>(v_new + src));
                const uint32_t kw[2] = {kb.x, kb.y}, vw[2] = {vb.x, vb.y};
                uint32_t k16[2], v16[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    k16[i] = e4m3x2_rn_sat(__fdiv_rn(__uint_as_float(kw[i] << 16), sc.x),
                                           __fdiv_rn(__uint_as_float(kw[i] & 0xFFFF0000u), sc.x));
                    v16[i] = e4m3x2_rn_sat(__fdiv_rn(__uint_as_float(vw[i] << 16), sc.y),
                                           __fdiv_rn(__uint_as_float(vw[i] & 0xFFFF0000u), sc.y));
                }
                *reinterpret_cast<uint32_t*>(k_cache + dst) = k16[0] | (k16[1] << 16);
                *reinterpret_cast<uint32_t*>(v_cache + dst) = v16[0] | (v16[1] << 16);
            } else {
                const uint4 kb = __ldcs(reinterpret_cast<const uint4*>(k_new + src));
                const uint4 vb = __ldcs(reinterpret_cast<const uint4*>(v_new + src));
                const uint32_t kw[4] = {kb.x, kb.y, kb.z, kb.w}, vw[4] = {vb.x, vb.y, vb.z, vb.w};
                uint32_t k16[4], v16[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    k16[i] = e4m3x2_rn_sat(__fdiv_rn(__uint_as_float(kw[i] << 16), sc.x),
                                           __fdiv_rn(__uint_as_float(kw[i] & 0xFFFF0000u), sc.x));
                    v16[i] = e4m3x2_rn_sat(__fdiv_rn(__uint_as_float(vw[i] << 16), sc.y),
                                           __fdiv_rn(__uint_as_float(vw[i] & 0xFFFF0000u), sc.y));
                }
                *reinterpret_cast<uint2*>(k_cache + dst) =
                    make_uint2(k16[0] | (k16[1] << 16), k16[2] | (k16[3] << 16));
                *reinterpret_cast<uint2*>(v_cache + dst) =
                    make_uint2(v16[0] | (v16[1] << 16), v16[2] | (v16[3] << 16));
            }
        }
    }
}

}  // namespace
}  // namespace yoco

extern "C" yoco_status_t yoco_kv_append(const void* k_new, const void* v_new, void* k_cache,
                                        void* v_cache, const int32_t* block_table,
                                        int32_t max_blocks_per_req, const int32_t* seq_lens,
                                        const int32_t* query_start_loc, int32_t num_reqs,
                                        int32_t num_tokens, int32_t num_blocks,
                                        int32_t block_size, int32_t num_kv_heads,
                                        int32_t head_dim, yoco_dtype_t dtype, int32_t* err_word,
                                        void* stream) {
    using namespace yoco;
    if (!dtype_ok(dtype)) return YOCO_ERR_UNSUPPORTED;
    if (!head_dim_ok(head_dim) || !block_size_ok(block_size)) return YOCO_ERR_UNSUPPORTED;
    if (num_reqs < 0 || num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 ||
        max_blocks_per_req <= 0)
        return YOCO_ERR_INVALID_ARG;
    if (num_tokens == 0 || num_reqs == 0) return YOCO_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !seq_lens || !query_start_loc)
        return YOCO_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return YOCO_ERR_INVALID_ARG;
    const int vecs = static_cast<int>(head_dim * elem_size(dtype) / 16);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (vecs) {
        case 8: e = launch_append<8>(k_new, v_new, k_cache, v_cache, block_table,
                                     max_blocks_per_req, seq_lens, query_start_loc, num_reqs,
                                     num_tokens, num_blocks, block_size, num_kv_heads, err_word, s);
            break;
        case 16: e = launch_append<16>(k_new, v_new, k_cache, v_cache, block_table,
                                       max_blocks_per_req, seq_lens, query_start_loc, num_reqs,
                                       num_tokens, num_blocks, block_size, num_kv_heads, err_word,
                                       s);
            break;
        case 32: e = launch_append<32>(k_new, v_new, k_cache, v_cache, block_table,
                                       max_blocks_per_req, seq_lens, query_start_loc, num_reqs,
                                       num_tokens, num_blocks, block_size, num_kv_heads, err_word,
                                       s);
            break;
        case 64: e = launch_append<64>(k_new, v_new, k_cache, v_cache, block_table,
                                       max_blocks_per_req, seq_lens, query_start_loc, num_reqs,
                                       num_tokens, num_blocks, block_size, num_kv_heads, err_word,
                                       s);
            break;
        default: return YOCO_ERR_UNSUPPORTED;
    }
    return cuda_status(e);
}

extern "C" yoco_status_t yoco_kv_append_e4m3(const void* k_new, const void* v_new, void* k_cache,
                                             void* v_cache, const float* page_scales,
                                             const int32_t* block_table,
                                             int32_t max_blocks_per_req, const int32_t* seq_lens,
                                             const int32_t* query_start_loc, int32_t num_reqs,
                                             int32_t num_tokens, int32_t num_blocks,
                                             int32_t block_size, int32_t num_kv_heads,
                                             int32_t head_dim, int32_t* err_word, void* stream) {
    using namespace yoco;
    if ((head_dim != 128 && head_dim != 256) || !block_size_ok(block_size))
        return YOCO_ERR_UNSUPPORTED;
    if (num_reqs < 0 || num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 ||
        max_blocks_per_req <= 0)
        return YOCO_ERR_INVALID_ARG;
    if (num_tokens == 0 || num_reqs == 0) return YOCO_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !page_scales || !block_table || !seq_lens ||
        !query_start_loc)
        return YOCO_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned16(page_scales))
        return YOCO_ERR_INVALID_ARG;
    int64_t blocks = (static_cast<int64_t>(num_tokens) + kAppendWarps - 1) / kAppendWarps;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const auto* kn = static_cast<const __nv_bfloat16*>(k_new);
    const auto* vn = static_cast<const __nv_bfloat16*>(v_new);
    auto* kc = static_cast<uint8_t*>(k_cache);
    auto* vc = static_cast<uint8_t*>(v_cache);
    const auto* sc = reinterpret_cast<const float4*>(page_scales);
    if (head_dim == 128)
        kv_append_e4m3_kernel<128><<<static_cast<unsigned>(blocks), kAppendWarps * 32, 0, s>>>(
            kn, vn, kc, vc, sc, block_table, max_blocks_per_req, seq_lens, query_start_loc,
            num_reqs, num_tokens, num_blocks, block_size, num_kv_heads, err_word);
    else
        kv_append_e4m3_kernel<256><<<static_cast<unsigned>(blocks), kAppendWarps * 32, 0, s>>>(
            kn, vn, kc, vc, sc, block_table, max_blocks_per_req, seq_lens, query_start_loc,
            num_reqs, num_tokens, num_blocks, block_size, num_kv_heads, err_word);
    return cuda_status(cudaGetLastError());
}
