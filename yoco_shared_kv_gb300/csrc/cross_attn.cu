// C entry points of the cross-decoder attention: argument checks, the split
// plan of the fp32 path, the pools' TMA descriptors and the launch.
//
// bf16 runs on the persistent tensor-core path (attn_tc.cu), an e4m3 cache
// on the same path with one-byte pages (attn_tc_e4m3.cu); fp32 runs on the
// CUDA-core split-KV path (attn_cc.cu).
#include <mutex>

#include "attn_common.cuh"

namespace yoco {
namespace {

constexpr int kCcWarpsHost = 4;

struct Plan {
    bool tc;          // tensor-core bf16 path
    int hb;           // CUDA-core path: query heads per CTA
    int split_pages;  // CUDA-core path: logical pages per split
    int max_splits;
    size_t ws_bytes;
};

bool make_plan(yoco_dtype_t dt, int max_rows, int H_q, int H_kv, int D, int BS, int max_seq_len,
               Plan& pl) {
    const bool e4m3 = dt == YOCO_E4M3;
    if (!(dtype_ok(dt) || e4m3) || !head_dim_ok(D) || !block_size_ok(BS)) return false;
    if (e4m3 && D == 64) return false;  // e4m3 pages need 128-byte rows
    if (H_q <= 0 || H_kv <= 0 || H_q % H_kv != 0 || H_q / H_kv > 16) return false;
    if (max_rows < 0 || max_seq_len <= 0) return false;
    const int G = H_q / H_kv;
    const int sms = device_sm_count();
    pl.tc = (dt == YOCO_BF16 || e4m3);
    pl.hb = 1;
    pl.split_pages = 0;
    pl.max_splits = 1;
    if (pl.tc) {
        pl.ws_bytes = tc_workspace_bytes(sms, H_kv, G, D, BS, e4m3);
        return true;
    }
    for (int c : {8, 4, 2, 1})
        if (G % c == 0) {
            pl.hb = c;
            break;
        }
    const int units = H_q / pl.hb;
    const int64_t pages_max = (static_cast<int64_t>(max_seq_len) + BS - 1) / BS;
    const int64_t target = 8ll * sms;  // CTAs to aim for at the longest row
    const int64_t unit_total = static_cast<int64_t>(max_rows > 0 ? max_rows : 1) * units;
    const int64_t want = (target + unit_total - 1) / unit_total;
    int64_t sp = (pages_max + want - 1) / want;
    const int64_t min_pages = kCcWarpsHost * 8;
    if (sp < min_pages) sp = min_pages;
    sp = (sp + kCcWarpsHost - 1) / kCcWarpsHost * kCcWarpsHost;
    if (sp > (1ll << 30)) return false;
    pl.split_pages = static_cast<int>(sp);
    pl.max_splits = static_cast<int>((pages_max + sp - 1) / sp);
    if (pl.max_splits > 65535) return false;
    pl.ws_bytes = pl.max_splits > 1 ? static_cast<size_t>(max_rows) * H_q * pl.max_splits *
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

// Pool [num_blocks * H_kv * BS rows][D] as a 2-D tensor of bf16 (esz 2) or
// bytes (esz 1); box = 128 bytes x BS rows with the 128-byte swizzle.
bool encode_pool(CUtensorMap* map, const void* pool, int64_t rows, int D, int BS, int esz) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * esz};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esz), static_cast<cuuint32_t>(BS)};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType ty =
        esz == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    return fn(map, ty, 2, const_cast<void*>(pool), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Small cache of encoded pool descriptors: the pools of a serving engine are
// fixed, so each is encoded once instead of on every call.
bool pool_map(CUtensorMap* map, const void* pool, int64_t rows, int D, int BS, int esz) {
    struct Entry {
        const void* pool;
        int64_t rows;
        int D, BS, esz, dev;
        CUtensorMap map;
    };
    static Entry cache[16];
    static int used = 0, next = 0;
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < used; ++i)
            if (cache[i].pool == pool && cache[i].rows == rows && cache[i].D == D &&
                cache[i].BS == BS && cache[i].esz == esz && cache[i].dev == dev) {
                *map = cache[i].map;
                return true;
            }
    }
    if (!encode_pool(map, pool, rows, D, BS, esz)) return false;
    std::lock_guard<std::mutex> lock(mu);
    Entry& e = cache[next];
    e.pool = pool;
    e.rows = rows;
    e.D = D;
    e.BS = BS;
    e.esz = esz;
    e.dev = dev;
    e.map = *map;
    next = (next + 1) % 16;
    if (used < 16) ++used;
    return true;
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

namespace yoco {
namespace {

// Shared body of the attention entry points; dtype YOCO_E4M3 = bf16 queries
// over an e4m3 cache with its scale records.
yoco_status_t run_attn(const void* q, const void* k_cache, const void* v_cache,
                       const float* page_scales, void* out, const int32_t* block_table,
                       int32_t max_blocks_per_req, const int32_t* seq_lens,
                       const int32_t* cross_query_start_loc, int32_t num_reqs, int32_t max_rows,
                       int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale,
                       yoco_dtype_t dtype, uint32_t flags, void* workspace,
                       size_t workspace_bytes, int32_t* err_word, void* stream,
                       const void* k_new = nullptr, const void* v_new = nullptr,
                       bool plan_only = false) {
    const bool e4m3 = dtype == YOCO_E4M3;
    if (flags & ~static_cast<uint32_t>(YOCO_ATTN_REVERSE | YOCO_ATTN_OVERLAP |
                                       YOCO_ATTN_KEEP_TAIL | YOCO_ATTN_PLANNED))
        return YOCO_ERR_INVALID_ARG;
    if (!(dtype_ok(dtype) || e4m3) || !head_dim_ok(head_dim) || !block_size_ok(block_size) ||
        (e4m3 && head_dim == 64))
        return YOCO_ERR_UNSUPPORTED;
    if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return YOCO_ERR_INVALID_ARG;
    if (num_q_heads / num_kv_heads > 16) return YOCO_ERR_UNSUPPORTED;
    if (num_reqs < 0 || max_rows < 0 || max_seq_len <= 0 || num_blocks <= 0 ||
        max_blocks_per_req <= 0 || !(scale > 0.f) || max_rows > 0x7fffffff / num_q_heads)
        return YOCO_ERR_INVALID_ARG;
    if (num_reqs == 0 || max_rows == 0) return YOCO_OK;
    if (!block_table || !seq_lens || !cross_query_start_loc) return YOCO_ERR_INVALID_ARG;
    if (!plan_only) {
        if (!q || !k_cache || !v_cache || !out) return YOCO_ERR_INVALID_ARG;
        if (e4m3 && (page_scales == nullptr || !aligned16(page_scales)))
            return YOCO_ERR_INVALID_ARG;
        if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
            return YOCO_ERR_INVALID_ARG;
    }
    if (workspace && !aligned16(workspace)) return YOCO_ERR_INVALID_ARG;
    // TMA row coordinates are signed 32-bit
    if (static_cast<int64_t>(num_blocks) * num_kv_heads * block_size > 0x7fffffffll)
        return YOCO_ERR_UNSUPPORTED;
    Plan pl;
    if (!make_plan(dtype, max_rows, num_q_heads, num_kv_heads, head_dim, block_size, max_seq_len,
                   pl))
        return YOCO_ERR_UNSUPPORTED;
    if (plan_only && !pl.tc) return YOCO_OK;  // the fp32 path plans its split grid on the host
    if (pl.ws_bytes > 0 && (workspace == nullptr || workspace_bytes < pl.ws_bytes))
        return YOCO_ERR_WORKSPACE;

    AttnParams p;
    p.q = q;
    p.out = out;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.cqsl = cross_query_start_loc;
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_pool = const_cast<void*>(k_cache);
    p.v_pool = const_cast<void*>(v_cache);
    p.err = err_word;
    p.max_blocks = max_blocks_per_req;
    p.num_reqs = num_reqs;
    p.max_rows = max_rows;
    p.H_q = num_q_heads;
    p.H_kv = num_kv_heads;
    p.G = num_q_heads / num_kv_heads;
    p.num_blocks = num_blocks;
    p.block_size = block_size;
    p.split_pages = pl.split_pages;
    p.max_splits = pl.max_splits;
    p.max_seq_len = max_seq_len;
    p.scales = reinterpret_cast<const float4*>(page_scales);
    p.scale_log2 = scale * kLog2e;
    p.reverse = (flags & YOCO_ATTN_REVERSE) ? 1 : 0;
    p.overlap = (flags & YOCO_ATTN_OVERLAP) ? 1 : 0;
    p.keep_tail = (flags & YOCO_ATTN_KEEP_TAIL) ? 1 : 0;
    // Tensor-core paths: the cross rows of a request (several when max_rows
    // exceeds num_reqs: chunked prefill, speculative verification) share one
    // walk over the request's pages in groups of rows whose heads fill the
    // kernel's head tile: one 8-wide tile when the rows per request (bounded
    // by max_rows / num_reqs) fit in it, else two (16 virtual heads). Partial
    // slots of grouped launches hold a full tile, those of one-row launches
    // the G heads; NT = 2 tiles run when the slot is wider than 8.
    {
        const int G = num_q_heads / num_kv_heads;
        const int64_t per_req = (static_cast<int64_t>(max_rows) + num_reqs - 1) / num_reqs;
        p.rg = 1;
        p.vhs = G;
        if (pl.tc && per_req > 1 && G <= 8) {
            if (G <= 4 && per_req <= 8 / G) {
                p.rg = 8 / G;
                p.vhs = 8;
            } else {
                p.rg = 16 / G;
                p.vhs = 16;
            }
        }
    }
    p.planned = (flags & YOCO_ATTN_PLANNED) ? 1 : 0;
    p.plan_only = plan_only ? 1 : 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (pl.tc) {
        p.ws_o = static_cast<float*>(workspace);  // carved up by the kernels (plan first)
        p.ws_ml = nullptr;
        CUtensorMap mk = {}, mv = {};
        const int64_t rows = static_cast<int64_t>(num_blocks) * num_kv_heads * block_size;
        const int esz = e4m3 ? 1 : 2;
        if (!plan_only && (!pool_map(&mk, k_cache, rows, head_dim, block_size, esz) ||
                           !pool_map(&mv, v_cache, rows, head_dim, block_size, esz)))
            return cuda_status(cudaErrorInvalidValue);  // descriptor encoding refused
        e = e4m3 ? launch_attn_tc_e4m3(mk, mv, p, head_dim, block_size, device_sm_count(), s)
                 : launch_attn_tc(mk, mv, p, head_dim, block_size, device_sm_count(), s);
    } else {
        p.ws_o = static_cast<float*>(workspace);
        p.ws_ml = pl.max_splits > 1
                      ? reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) +
                                                  static_cast<size_t>(max_rows) * num_q_heads *
                                                      pl.max_splits * head_dim * 4)
                      : nullptr;
        e = launch_attn_cc(k_cache, v_cache, p, head_dim, pl.hb, s);
    }
    return cuda_status(e);
}

}  // namespace
}  // namespace yoco

extern "C" yoco_status_t yoco_cross_attn_paged(
    const void* q, const void* k_cache, const void* v_cache, void* out, const int32_t* block_table,
    int32_t max_blocks_per_req, const int32_t* seq_lens, const int32_t* cross_query_start_loc,
    int32_t num_reqs, int32_t max_rows, int32_t max_seq_len, int32_t num_q_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale,
    yoco_dtype_t dtype, uint32_t flags, void* workspace, size_t workspace_bytes, int32_t* err_word,
    void* stream) {
    if (dtype == YOCO_E4M3) return YOCO_ERR_UNSUPPORTED;  // the e4m3 cache has its own entry
    return yoco::run_attn(q, k_cache, v_cache, nullptr, out, block_table, max_blocks_per_req,
                          seq_lens, cross_query_start_loc, num_reqs, max_rows, max_seq_len,
                          num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                          dtype, flags, workspace, workspace_bytes, err_word, stream);
}

extern "C" yoco_status_t yoco_cross_attn_plan(
    const int32_t* block_table, int32_t max_blocks_per_req, const int32_t* seq_lens,
    const int32_t* cross_query_start_loc, int32_t num_reqs, int32_t max_rows, int32_t max_seq_len,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
    int32_t num_blocks, yoco_dtype_t dtype, uint32_t flags, void* workspace,
    size_t workspace_bytes, int32_t* err_word, void* stream) {
    if (flags & ~static_cast<uint32_t>(YOCO_ATTN_OVERLAP)) return YOCO_ERR_INVALID_ARG;
    return yoco::run_attn(nullptr, nullptr, nullptr, nullptr, nullptr, block_table,
                          max_blocks_per_req, seq_lens, cross_query_start_loc, num_reqs, max_rows,
                          max_seq_len, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                          1.0f, dtype, flags, workspace, workspace_bytes, err_word, stream, nullptr,
                          nullptr, true);
}

extern "C" yoco_status_t yoco_cross_attn_paged_e4m3(
    const void* q, const void* k_cache, const void* v_cache, const float* page_scales, void* out,
    const int32_t* block_table, int32_t max_blocks_per_req, const int32_t* seq_lens,
    const int32_t* cross_query_start_loc, int32_t num_reqs, int32_t max_rows, int32_t max_seq_len,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
    int32_t num_blocks, float scale, uint32_t flags, void* workspace, size_t workspace_bytes,
    int32_t* err_word, void* stream) {
    return yoco::run_attn(q, k_cache, v_cache, page_scales, out, block_table, max_blocks_per_req,
                          seq_lens, cross_query_start_loc, num_reqs, max_rows, max_seq_len,
                          num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                          YOCO_E4M3, flags, workspace, workspace_bytes, err_word, stream);
}

extern "C" yoco_status_t yoco_cross_decode_step(
    const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
    const float* page_scales, void* out, const int32_t* block_table, int32_t max_blocks_per_req,
    const int32_t* seq_lens, const int32_t* query_start_loc, int32_t num_reqs,
    int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, int32_t num_blocks, float scale, yoco_dtype_t dtype, uint32_t flags,
    void* workspace, size_t workspace_bytes, int32_t* err_word, void* stream) {
    using namespace yoco;
    if (dtype != YOCO_BF16 && dtype != YOCO_E4M3) return YOCO_ERR_UNSUPPORTED;
    if (num_reqs > 0 && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)))
        return YOCO_ERR_INVALID_ARG;
    if (flags & YOCO_ATTN_REVERSE) return YOCO_ERR_INVALID_ARG;  // the fused step walks forward
    // decode: one new token and one cross row per request, so query_start_loc is
    // also the cross query_start_loc and num_reqs bounds the rows
    return run_attn(q, k_cache, v_cache, dtype == YOCO_E4M3 ? page_scales : nullptr, out,
                    block_table, max_blocks_per_req, seq_lens, query_start_loc, num_reqs,
                    num_reqs, max_seq_len, num_q_heads, num_kv_heads, head_dim, block_size,
                    num_blocks, scale, dtype, flags, workspace, workspace_bytes, err_word, stream,
                    k_new, v_new);
}
