// Shared definitions of the cross-decoder attention kernels (internal).
#pragma once

#include "common.cuh"

namespace yoco {

// Launch parameters common to both attention paths.
struct AttnParams {
    const void* q;              // [max_rows][H_q][D]
    void* out;                  // [max_rows][H_q][D]
    const int32_t* block_table; // [num_reqs][max_blocks]
    const int32_t* seq_lens;    // [num_reqs]
    const int32_t* cqsl;        // [num_reqs + 1] cross query_start_loc
    // fused decode step (tensor-core paths): this step's new K^/V^ rows, bf16
    // [num_reqs][H_kv][D] (one token per request), appended to the pools by the
    // same launch; null otherwise
    const void* k_new;
    const void* v_new;
    void* k_pool;
    void* v_pool;
    float* ws_o;                // partial outputs (layout depends on the path)
    float2* ws_ml;              // partial (running max in log2 units, sum)
    int32_t* err;
    int32_t max_blocks;
    int32_t num_reqs;
    int32_t max_rows;
    int32_t H_q, H_kv, G;
    int32_t num_blocks;
    int32_t block_size;
    int32_t split_pages;        // CUDA-core path: logical pages per split
    int32_t max_splits;         // CUDA-core path
    int32_t max_seq_len;        // host bound on seq_lens (the CUDA-core split plan is sized by it)
    const float4* scales;       // e4m3 cache: {k_scale, v_scale, -, -} per (page, kv head)
    float scale_log2;           // softmax scale * log2(e)
    int32_t reverse;            // tensor-core path: walk each worker's pages from the end
    int32_t overlap;            // tensor-core path: launch as a programmatic dependent
    int32_t keep_tail;          // tensor-core path: L2 hints, keep this walk's tail for the next layer
    int32_t rg;                 // tensor-core path: cross rows of a request grouped on one walk (1: none)
    int32_t vhs;                // tensor-core path: virtual heads (group rows x heads) per partial slot
    int32_t planned;            // tensor-core path: the workspace already holds this step's plan
    int32_t plan_only;          // tensor-core path: make the plan, launch no attention
};

// Wait limit for one asynchronous page copy before a kernel gives up.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ bool launch_aborted(const AttnParams& p) {
    return p.err != nullptr &&
           (*reinterpret_cast<volatile int32_t*>(p.err) & YOCO_DEVERR_TIMEOUT) != 0;
}

template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ float from_float<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Host-side launchers (one per path). `tc_workspace_bytes` / `cc_*` give the
// scratch each path needs.
size_t tc_workspace_bytes(int sms, int H_kv, int G, int D, int BS, bool e4m3);
int tc_ctas(int sms);
cudaError_t launch_attn_tc(const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p,
                           int D, int BS, int sms, cudaStream_t s);
cudaError_t launch_attn_tc_e4m3(const CUtensorMap& mk, const CUtensorMap& mv,
                                const AttnParams& p, int D, int BS, int sms, cudaStream_t s);
cudaError_t launch_attn_cc(const void* k_cache, const void* v_cache, const AttnParams& p, int D,
                           int hb, cudaStream_t s);

}  // namespace yoco
