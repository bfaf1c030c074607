// Library-wide C entry points: status strings, version, L2 persistence window.
#include "common.cuh"

extern "C" const char* yoco_status_string(yoco_status_t status) {
    switch (status) {
        case YOCO_OK: return "ok";
        case YOCO_ERR_INVALID_ARG: return "invalid argument";
        case YOCO_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case YOCO_ERR_WORKSPACE: return "workspace missing or too small";
        case YOCO_ERR_CUDA: return "CUDA runtime error";
    }
    return "unknown status";
}

extern "C" int32_t yoco_version(void) { return 100; }  // 0.1.0

namespace yoco {
namespace {
thread_local int g_last_cuda_error = 0;
}
yoco_status_t cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return YOCO_OK;
    g_last_cuda_error = static_cast<int>(e);
    return YOCO_ERR_CUDA;
}
}  // namespace yoco

extern "C" int32_t yoco_last_cuda_error(void) { return yoco::g_last_cuda_error; }

extern "C" const char* yoco_last_cuda_error_string(void) {
    return cudaGetErrorString(static_cast<cudaError_t>(yoco::g_last_cuda_error));
}

// The serial cross-decoder layers re-read one shared cache ("YOCO
// 论文与推理数据流详解" §11); when the cache (or its hot part) fits in L2,
// a persisting access-policy window keeps it there between layers.
extern "C" yoco_status_t yoco_set_l2_window(void* stream, void* base, size_t bytes,
                                            float hit_ratio) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStreamAttrValue attr = {};
    if (bytes == 0 || base == nullptr) {
        attr.accessPolicyWindow.base_ptr = nullptr;
        attr.accessPolicyWindow.num_bytes = 0;
        attr.accessPolicyWindow.hitRatio = 0.f;
        attr.accessPolicyWindow.hitProp = cudaAccessPropertyNormal;
        attr.accessPolicyWindow.missProp = cudaAccessPropertyNormal;
        YOCO_CUDA_OK(cudaStreamSetAttribute(s, cudaStreamAttributeAccessPolicyWindow, &attr));
        // lines already marked persisting would otherwise keep their set-aside,
        // and the set-aside itself (this context's only) goes back to none
        YOCO_CUDA_OK(cudaCtxResetPersistingL2Cache());
        YOCO_CUDA_OK(cudaDeviceSetLimit(cudaLimitPersistingL2CacheSize, 0));
        return YOCO_OK;
    }
    if (!(hit_ratio <= 1.f)) return YOCO_ERR_INVALID_ARG;  // negative: automatic
    int dev = 0, max_win = 0, max_persist = 0;
    YOCO_CUDA_OK(cudaGetDevice(&dev));
    YOCO_CUDA_OK(cudaDeviceGetAttribute(&max_win, cudaDevAttrMaxAccessPolicyWindowSize, dev));
    YOCO_CUDA_OK(cudaDeviceGetAttribute(&max_persist, cudaDevAttrMaxPersistingL2CacheSize, dev));
    if (max_win <= 0 || max_persist <= 0) return YOCO_ERR_UNSUPPORTED;
    const size_t win = bytes < static_cast<size_t>(max_win) ? bytes : static_cast<size_t>(max_win);
    const size_t keep = win < static_cast<size_t>(max_persist) ? win : static_cast<size_t>(max_persist);
    // the set-aside is a limit of this process's context only
    YOCO_CUDA_OK(cudaDeviceSetLimit(cudaLimitPersistingL2CacheSize, keep));
    attr.accessPolicyWindow.base_ptr = base;
    attr.accessPolicyWindow.num_bytes = win;
    // automatic ratio: as many of the window's lines as the set-aside holds
    attr.accessPolicyWindow.hitRatio =
        hit_ratio < 0.f ? static_cast<float>(static_cast<double>(keep) / static_cast<double>(win))
                        : hit_ratio;
    attr.accessPolicyWindow.hitProp = cudaAccessPropertyPersisting;
    attr.accessPolicyWindow.missProp = cudaAccessPropertyStreaming;
    YOCO_CUDA_OK(cudaStreamSetAttribute(s, cudaStreamAttributeAccessPolicyWindow, &attr));
    return YOCO_OK;
}

namespace yoco {
namespace {
// One thread arms a barrier for bytes that no copy will deliver and waits on
// it with the same bounded helper the attention kernel uses.
__global__ void selftest_wait_kernel(int32_t* err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar, 1024);  // no copy is issued: the phase never completes
    if (!mbar_wait_bounded(&bar, 0, limit_ns)) set_err(err, YOCO_DEVERR_TIMEOUT);
}
}  // namespace
}  // namespace yoco

extern "C" yoco_status_t yoco_selftest_wait_timeout(int32_t* err_word, uint32_t limit_us,
                                                    void* stream) {
    if (err_word == nullptr || limit_us == 0 || limit_us > 2000000u) return YOCO_ERR_INVALID_ARG;
    yoco::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        err_word, static_cast<uint64_t>(limit_us) * 1000ull);
    return yoco::cuda_status(cudaGetLastError());
}

// Traffic model: the algorithmic bytes one cross-decoder step moves per request.
extern "C" int64_t yoco_cross_decoder_bytes(const int32_t* query_start_loc,
                                            const int32_t* rows_per_req, const int32_t* seq_lens,
                                            int32_t num_reqs, int32_t layers, int32_t num_q_heads,
                                            int32_t num_kv_heads, int32_t head_dim,
                                            int32_t block_size, yoco_dtype_t dtype,
                                            int64_t* per_req_bytes) {
    const bool e4m3 = dtype == YOCO_E4M3;
    if (num_reqs < 0 || layers < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || !(yoco::dtype_ok(dtype) || e4m3))
        return -1;
    if (num_reqs > 0 && (query_start_loc == nullptr || seq_lens == nullptr)) return -1;
    // e4m3: one-byte keys/values, bf16 queries/outputs, a 16-byte scale record per page
    const int64_t elem = e4m3 ? 2 : static_cast<int64_t>(yoco::elem_size(dtype));
    const int64_t kv_elem = e4m3 ? 1 : elem;
    const int64_t page_meta = 4 + (e4m3 ? 16 : 0);
    int64_t total = 0;
    for (int32_t r = 0; r < num_reqs; ++r) {
        const int64_t q_len = static_cast<int64_t>(query_start_loc[r + 1]) - query_start_loc[r];
        const int64_t want = rows_per_req ? rows_per_req[r] : 1;
        if (q_len < 0 || want < 0) return -1;
        const int64_t k = want < q_len ? want : q_len;
        int64_t b = 0;
        if (k > 0) {
            // the rows of a request share its pages: they are read once, up to
            // the last row's causal end (seq_len keys); each row has its own
            // query and output
            int64_t kv = seq_lens[r];
            if (kv < 0) kv = 0;
            b = kv * 2 * num_kv_heads * head_dim * kv_elem + k * 2ll * num_q_heads * head_dim * elem +
                page_meta * ((kv + block_size - 1) / block_size) * num_kv_heads;
        }
        b *= layers;
        if (per_req_bytes) per_req_bytes[r] = b;
        total += b;
    }
    return total;
}
