// yoco_cross_attn_paged_noalloc: the cross-decoder attention with its
// scratch in a fixed device array owned by this library, for callers that
// cannot allocate device memory.
//
// Who cannot allocate: code that runs while a CUDA graph is being captured
// (cudaMalloc is not allowed there), engines whose device memory is carved
// out once at start-up and handed out by their own allocator (an inference
// server that forbids allocations after warm-up), and hosts embedding this
// library through a C plugin interface that offers no allocator at all.
// They pass inputs and outputs as usual; the split-KV partial results live
// in the array below instead of a caller-provided workspace.
//
// The array is a file-scope __device__ variable: every GPU on which this
// library's module is loaded holds kStaticScratchBytes of it until the
// process exits. Host code must not use its name as a pointer (that is a
// host-side stand-in); the device address is looked up once per device
// with cudaGetSymbolAddress.
#include <mutex>

#include "common.cuh"

namespace yoco {
namespace {

constexpr size_t kStaticScratchBytes = 16u << 20;  // 16 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_attn_scratch[kStaticScratchBytes];

// Device address of g_attn_scratch on the current device, looked up on the
// first call per device (that call must come before any stream capture).
cudaError_t scratch_address(void** out) {
    static void* addr[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attn_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *out = addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace yoco

extern "C" size_t yoco_cross_attn_noalloc_capacity(void) { return yoco::kStaticScratchBytes; }

extern "C" yoco_status_t yoco_cross_attn_paged_noalloc(
    const void* q, const void* k_cache, const void* v_cache, void* out, const int32_t* block_table,
    int32_t max_blocks_per_req, const int32_t* seq_lens, const int32_t* cross_query_start_loc,
    int32_t num_reqs, int32_t max_rows, int32_t max_seq_len, int32_t num_q_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale,
    yoco_dtype_t dtype, int32_t* err_word, void* stream) {
    using namespace yoco;
    // the e4m3 cache has its own entry; refuse it (and unknown dtypes) before any CUDA call
    if (!dtype_ok(dtype)) return YOCO_ERR_UNSUPPORTED;
    const size_t need = yoco_cross_attn_workspace_size(max_rows, num_q_heads, num_kv_heads,
                                                       head_dim, block_size, max_seq_len, dtype);
    if (need > kStaticScratchBytes) return YOCO_ERR_WORKSPACE;  // more than the fixed array holds
    void* scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) return cuda_status(e);
    // Every scratch word a launch reads is written earlier in that same
    // launch, so nothing needs clearing between calls.
    return yoco_cross_attn_paged(q, k_cache, v_cache, out, block_table, max_blocks_per_req,
                                 seq_lens, cross_query_start_loc, num_reqs, max_rows,
                                 max_seq_len, num_q_heads, num_kv_heads, head_dim, block_size,
                                 num_blocks, scale, dtype, 0u, scratch, kStaticScratchBytes,
                                 err_word, stream);
}
