// Device helpers shared by the library's kernels (sm_103a).
//
// Thin inline-PTX wrappers around the asynchronous-copy, barrier and
// warp-level matrix instructions the kernels use, plus the host-side status
// plumbing. Nothing here is specific to one kernel.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "yoco_kv.h"

namespace yoco {

// ---------------------------------------------------------------- host side

// Maps a CUDA runtime result to a status, remembering a failure for
// yoco_last_cuda_error() on this thread.
yoco_status_t cuda_status(cudaError_t e);

#define YOCO_CUDA_OK(expr)                                \
    do {                                                  \
        cudaError_t e_ = (expr);                          \
        if (e_ != cudaSuccess) return yoco::cuda_status(e_); \
    } while (0)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t elem_size(yoco_dtype_t dt) { return dt == YOCO_BF16 ? 2 : 4; }

inline bool dtype_ok(yoco_dtype_t dt) { return dt == YOCO_F32 || dt == YOCO_BF16; }

inline bool head_dim_ok(int d) { return d == 64 || d == 128 || d == 256; }

inline bool block_size_ok(int b) { return b == 16 || b == 32; }

// Number of SMs of the current device (queried each time; cheap attribute read).
int device_sm_count();

// ------------------------------------------------------------- device side

__device__ __forceinline__ void set_err(int32_t* err, int32_t bits) {
    if (err != nullptr) atomicOr(err, bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// mbarrier (CTA scope) ------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Makes barrier initialisation visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, giving up after `limit_ns`
// of wall time (and after a hard iteration cap). Returns false on give-up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1; it < (1u << 26); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// Orders this thread's generic-proxy shared-memory writes before later
// asynchronous-proxy (TMA) accesses of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// TMA: 2-D tiled tensor load global -> shared, completion on an mbarrier.
// x is the innermost coordinate (elements); the caller keeps x * elem_size
// a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// The same with an L2 cache-eviction policy (from make_l2_policy_*).
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int32_t x,
                                                 int32_t y, uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// L2 eviction policies for cache-hinted copies: keep the lines (evict last)
// or let them go first.
__device__ __forceinline__ uint64_t make_l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t make_l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Bulk (untiled) copy global -> shared, completion on an mbarrier. Both
// addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Asynchronous global -> shared copies of 16 / 8 bytes (both addresses
// aligned to the size), then a wait for every copy this thread issued.
__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src))
                 : "memory");
}
__device__ __forceinline__ void cp_async_8(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src))
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Named barrier of two warps (64 threads; id 1..15, 0 is __syncthreads). Both
// warps must reach it the same number of times.
__device__ __forceinline__ void pair_sync(int id) {
    asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
}

// The same barrier, returning the AND of the 64 threads' predicates: both
// warps leave with the same answer.
__device__ __forceinline__ bool pair_all(int id, bool v) {
    uint32_t r;
    asm volatile(
        "{ .reg .pred p, q;\n"
        "  setp.ne.u32 p, %1, 0;\n"
        "  bar.red.and.pred q, %2, 64, p;\n"
        "  selp.u32 %0, 1, 0, q; }"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "r"(id)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Warp-level matrix helpers ----------------------------------------------------

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A(16x16, row) * B(16x8, col) + D, f16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 b16 matrix held one packed pair per lane.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Two floats -> packed bf16x2, round to nearest even; `lo` in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t x) {
    return __uint_as_float(x & 0xFFFF0000u);
}

// Two floats -> packed f16x2, round to nearest even; `lo` in bits 0..15.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float f16lo_to_f32(uint32_t x) {
    float f;
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.f32.f16 %0, l; }" : "=f"(f) : "r"(x));
    return f;
}
__device__ __forceinline__ float f16hi_to_f32(uint32_t x) {
    float f;
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.f32.f16 %0, h; }" : "=f"(f) : "r"(x));
    return f;
}

// e4m3 -> f16 is exact (every e4m3 value is an f16 value): the two bytes of
// the low (lo_half) or high 16 bits of x become an f16x2, lower byte in the
// lower half.
__device__ __forceinline__ uint32_t e4m3x2_lo_to_f16x2(uint32_t x) {
    uint32_t r;
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.rn.f16x2.e4m3x2 %0, l; }" : "=r"(r) : "r"(x));
    return r;
}
__device__ __forceinline__ uint32_t e4m3x2_hi_to_f16x2(uint32_t x) {
    uint32_t r;
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.rn.f16x2.e4m3x2 %0, h; }" : "=r"(r) : "r"(x));
    return r;
}

// Scale records of the 8-bit cache: {k_scale, v_scale, -, -} per (page, kv head).
__device__ __forceinline__ bool scale_usable(float s) { return s > 0.f && s <= 3.4e38f; }

// Two floats -> two e4m3 codes (nearest, ties to even, saturating to +-448);
// `lo` in bits 0..7.
__device__ __forceinline__ uint32_t e4m3x2_rn_sat(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Eight bf16 values (two packed words each in a, b) -> eight e4m3 codes of
// value / scale (float32 division, the cache's quantisation rule), low byte first.
__device__ __forceinline__ uint2 quantise8_e4m3(uint4 a, float scale) {
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        c[i] = e4m3x2_rn_sat(__fdiv_rn(__uint_as_float(w[i] << 16), scale),
                             __fdiv_rn(__uint_as_float(w[i] & 0xFFFF0000u), scale));
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// 2^x with the hardware approximation (the softmax runs in the log2 domain).
__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr float kLog2e = 1.4426950408889634f;

// Row n of the cross batch -> (request, kv_len). Returns false when the row
// does not exist (n >= total rows). kv_len <= 0 signals an empty row.
__device__ __forceinline__ bool locate_row(const int32_t* __restrict__ cqsl, int32_t num_reqs,
                                           int32_t n, const int32_t* __restrict__ seq_lens,
                                           int32_t& req, int32_t& kv_len) {
    if (num_reqs <= 0 || n >= __ldg(cqsl + num_reqs)) return false;
    // first r with cqsl[r + 1] > n
    int32_t lo = 0, hi = num_reqs - 1;
    while (lo < hi) {
        const int32_t mid = (lo + hi) >> 1;
        if (__ldg(cqsl + mid + 1) > n) hi = mid;
        else lo = mid + 1;
    }
    const int32_t c0 = __ldg(cqsl + lo), c1 = __ldg(cqsl + lo + 1);
    req = lo;
    kv_len = __ldg(seq_lens + lo) - (c1 - c0) + (n - c0) + 1;
    return true;
}

}  // namespace yoco
