// yoco_select_cross_rows: compact a mixed prefill/decode batch to the
// cross-decoder rows.
//
// "You Only Cache Once, in vLLM", "Implementation in vLLM": at every
// scheduling step the cross-decoder only needs, per request, its last
// scheduled token (the last prompt token of a prefill, or the decode
// token); "Adding torch.compile and cudagraph support": the cross-decoder
// metadata gets per-request row counts, a new query_start_loc that is their
// running sum, and unchanged seq_lens / block table.
//
// Design: one CTA of 1024 threads walks the requests in chunks of 1024,
// each thread computes its request's row count k_r, a warp-shuffle scan plus
// a scan of the 32 warp totals gives the exclusive offsets, and a running
// carry links the chunks. Integer-only, so bit-exact; the row count stays on
// the device (no host synchronisation, unlike reading it back with .item()).
#include "common.cuh"

namespace yoco {
namespace {

constexpr int kSelectThreads = 1024;

__global__ void __launch_bounds__(kSelectThreads)
    select_rows_kernel(const int32_t* __restrict__ qsl, const int32_t* __restrict__ rows_per_req,
                       int32_t num_reqs, int32_t* __restrict__ rows, int32_t* __restrict__ cqsl,
                       int32_t* __restrict__ num_rows, int32_t* err) {
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t carry_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        carry_s = 0;
        cqsl[0] = 0;
    }
    __syncthreads();
    for (int32_t base = 0; base < num_reqs; base += kSelectThreads) {
        const int32_t r = base + tid;
        int32_t k = 0, end = 0;
        if (r < num_reqs) {
            end = __ldg(qsl + r + 1);
            const int32_t q_len = end - __ldg(qsl + r);
            const int32_t want = rows_per_req ? __ldg(rows_per_req + r) : 1;
            if (q_len < 0 || want < 0) set_err(err, YOCO_DEVERR_OFFSETS);
            else k = want < q_len ? want : q_len;
        }
        // inclusive scan of k within the warp
        int32_t incl = k;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int32_t t = warp_tot[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int32_t v = __shfl_up_sync(0xffffffffu, t, off);
                if (lane >= off) t += v;
            }
            warp_tot[lane] = t;  // inclusive over warps
        }
        __syncthreads();
        const int32_t carry = carry_s;
        const int32_t start = carry + (warp ? warp_tot[warp - 1] : 0) + incl - k;
        if (r < num_reqs) {
            cqsl[r + 1] = start + k;
            for (int32_t i = 0; i < k; ++i) rows[start + i] = end - k + i;
        }
        __syncthreads();
        if (tid == 0) carry_s = carry + warp_tot[31];
        __syncthreads();
    }
    if (tid == 0) *num_rows = carry_s;
}

}  // namespace
}  // namespace yoco

extern "C" yoco_status_t yoco_select_cross_rows(const int32_t* query_start_loc,
                                                const int32_t* rows_per_req, int32_t num_reqs,
                                                int32_t* row_indices,
                                                int32_t* cross_query_start_loc,
                                                int32_t* num_rows, int32_t* err_word,
                                                void* stream) {
    using namespace yoco;
    if (num_reqs < 0) return YOCO_ERR_INVALID_ARG;
    if (!query_start_loc || !cross_query_start_loc || !num_rows) return YOCO_ERR_INVALID_ARG;
    if (num_reqs > 0 && !row_indices) return YOCO_ERR_INVALID_ARG;
    select_rows_kernel<<<1, kSelectThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        query_start_loc, rows_per_req, num_reqs, row_indices, cross_query_start_loc, num_rows,
        err_word);
    return cuda_status(cudaGetLastError());
}
