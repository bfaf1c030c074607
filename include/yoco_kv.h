/*
 * yoco_kv.h — C ABI of the YOCO shared-KV cross-decoder hot path (GB300, sm_103a).
 *
 * A YOCO model computes one shared K^/V^ per token at the self-decoder
 * boundary and caches it once; every cross-decoder layer then attends from
 * its own queries to that one cache ("YOCO 论文与推理数据流详解", §3 and
 * §10.3–§10.4). In a continuous-batching engine only the last scheduled
 * token of each request has to enter the cross-decoder ("You Only Cache
 * Once, in vLLM", "Implementation in vLLM"). The three calls below are that
 * path: append the new K^/V^ into a paged cache, compact the batch to the
 * cross-decoder rows, and run causal paged GQA attention for one layer.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Pointers named *device* are CUDA device pointers; the caller owns all
 *    memory. The library never allocates, frees or synchronises a stream;
 *    work is enqueued on `stream` (0 = legacy default stream).
 *  - Host-detectable problems (null pointers, unsupported shapes, bad
 *    alignment, too-small workspace) return a status before anything is
 *    launched. A failed launch returns YOCO_ERR_CUDA.
 *  - Data-dependent problems found on the device (a page id outside
 *    [0, num_blocks), a position past the block table, a row with no key,
 *    malformed offsets) never trap: the offending element is skipped and the
 *    matching YOCO_DEVERR_* bit is OR-ed into `*err_word` (a device int32,
 *    may be NULL). The caller clears it and reads it when it wants.
 *  - Every call is asynchronous and makes no host<->device transfer, so a
 *    sequence of calls can be captured in a CUDA graph.
 *  - Cache layout ("KV cache memory systems", "Contiguous allocation wastes
 *    capacity": logical token blocks map through a block table to
 *    physical pages; the layout inside a page is not given there): two
 *    pools k_cache / v_cache of shape [num_blocks][num_kv_heads][block_size]
 *    [head_dim], row-major, so one (page, kv head) is one contiguous run of
 *    block_size * head_dim elements. Token position p of request r is page
 *    block_table[r * max_blocks_per_req + p / block_size], slot
 *    p % block_size.
 *  - Metadata names follow vLLM's CommonAttentionMetadata as shown in
 *    "You Only Cache Once, in vLLM": query_start_loc [num_reqs + 1] holds
 *    exclusive offsets of each request's scheduled tokens, seq_lens
 *    [num_reqs] the tokens in the cache after this step (the scheduled
 *    tokens included), block_table [num_reqs][max_blocks_per_req] int32.
 *  - Supported shapes: head_dim in {64, 128, 256}; block_size in {16, 32};
 *    num_q_heads a multiple of num_kv_heads with a group of at most 16;
 *    dtype YOCO_F32 or YOCO_BF16 (attention accumulates in fp32 and writes
 *    the input dtype).
 *  - Preconditions the library cannot see: a step must not append into a
 *    page another request still shares (prefix pages are copy-on-write,
 *    "KV cache memory systems", "Prefix caching needs identity rules"); rows
 *    skipped by the selection have no cross-decoder output, so a request
 *    that wants prompt log-probabilities must not use it ("You Only Cache
 *    Once, in vLLM", "Note").
 */
#ifndef YOCO_KV_H_
#define YOCO_KV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    YOCO_OK = 0,
    YOCO_ERR_INVALID_ARG = 1, /* null pointer, negative size, misaligned buffer, bad metadata shape */
    YOCO_ERR_UNSUPPORTED = 2, /* head_dim / block_size / group / dtype outside the supported set */
    YOCO_ERR_WORKSPACE = 3,   /* workspace pointer null or smaller than the size query returned */
    YOCO_ERR_CUDA = 4         /* a CUDA runtime call or kernel launch failed */
} yoco_status_t;

/* YOCO_E4M3 names the 8-bit cache of the *_e4m3 calls (bf16 queries and
 * outputs over an e4m3 cache); only yoco_cross_attn_workspace_size and
 * yoco_cross_decoder_bytes take it. */
typedef enum { YOCO_F32 = 0, YOCO_BF16 = 1, YOCO_E4M3 = 2 } yoco_dtype_t;

/* Flags of yoco_cross_attn_paged. */
#define YOCO_ATTN_REVERSE 0x1u /* tensor-core paths: walk each worker's pages last to first */
#define YOCO_ATTN_OVERLAP 0x2u /* tensor-core paths: may start while the previous kernel drains */
#define YOCO_ATTN_KEEP_TAIL 0x4u /* tensor-core paths: L2 hints that keep this walk's tail for the next layer */
#define YOCO_ATTN_PLANNED 0x8u /* tensor-core paths: the workspace holds this step's plan (yoco_cross_attn_plan) */

/* Bits OR-ed into *err_word by device code. */
#define YOCO_DEVERR_PAGE_RANGE 0x1   /* block_table entry outside [0, num_blocks) */
#define YOCO_DEVERR_POS_RANGE 0x2    /* position beyond max_blocks_per_req * block_size, or negative;
                                        attention: a row with more keys than max_seq_len */
#define YOCO_DEVERR_EMPTY_ROW 0x4    /* a cross row with no key to attend (seq_len < rows of its request) */
#define YOCO_DEVERR_OFFSETS 0x8      /* query_start_loc decreasing, or rows_per_req negative */
#define YOCO_DEVERR_TIMEOUT 0x10     /* a bounded wait on an asynchronous copy gave up */
#define YOCO_DEVERR_SCALE 0x20       /* e4m3 cache: a page scale outside the supported range */
#define YOCO_DEVERR_PLAN 0x40        /* YOCO_ATTN_PLANNED, but the workspace holds no plan for these shapes */

/*
 * yoco_kv_append — write the step's new shared K^/V^ into the paged cache.
 *
 * "YOCO 论文与推理数据流详解" §7.3 / §10.3: each token's K^/V^ is produced
 * once at the self-decoder boundary and appended once to the single global
 * cache (prefill appends the whole prompt, decode one position).
 *
 *   k_new, v_new      device, [num_tokens][num_kv_heads][head_dim], dtype; 16-byte aligned
 *   k_cache, v_cache  device pools, layout above; 16-byte aligned
 *   block_table       device int32 [num_reqs][max_blocks_per_req]
 *   seq_lens          device int32 [num_reqs]
 *   query_start_loc   device int32 [num_reqs + 1]; query_start_loc[num_reqs] must equal num_tokens
 *   err_word          device int32 or NULL
 * Token j of request r (0 <= j < q_len, q_len = qsl[r+1] - qsl[r]) goes to
 * position seq_lens[r] - q_len + j. Results are bit-exact copies.
 */
yoco_status_t yoco_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const int32_t* block_table, int32_t max_blocks_per_req,
                             const int32_t* seq_lens, const int32_t* query_start_loc,
                             int32_t num_reqs, int32_t num_tokens, int32_t num_blocks,
                             int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                             yoco_dtype_t dtype, int32_t* err_word, void* stream);

/*
 * yoco_select_cross_rows — compact a mixed prefill/decode batch to the
 * cross-decoder rows.
 *
 * "You Only Cache Once, in vLLM", "Implementation in vLLM": the cross-decoder
 * only needs the last prompt token of a prefilling request and every decode
 * token; its metadata builder ("Adding torch.compile and cudagraph support")
 * gives each request k_r rows, a new query_start_loc = running sum of k_r,
 * and keeps seq_lens and the block table unchanged.
 *
 *   query_start_loc        device int32 [num_reqs + 1]
 *   rows_per_req           device int32 [num_reqs] or NULL (= 1 per request);
 *                          k_r = min(rows_per_req[r], q_len_r)
 *   row_indices            device int32 out, capacity >= sum of k_r (<= num_tokens);
 *                          row_indices[cqsl[r] + i] = qsl[r+1] - k_r + i
 *   cross_query_start_loc  device int32 out [num_reqs + 1]
 *   num_rows               device int32 out [1] (= cross_query_start_loc[num_reqs])
 *   err_word               device int32 or NULL
 * Bit-exact. num_reqs may be 0. Runs as one CTA; no host synchronisation.
 */
yoco_status_t yoco_select_cross_rows(const int32_t* query_start_loc, const int32_t* rows_per_req,
                                     int32_t num_reqs, int32_t* row_indices,
                                     int32_t* cross_query_start_loc, int32_t* num_rows,
                                     int32_t* err_word, void* stream);

/*
 * yoco_cross_attn_workspace_size — bytes of fp32 scratch that
 * yoco_cross_attn_paged needs for these bounds on the current device (the
 * split-KV partial outputs and their log-sum-exp statistics). Returns 0 for
 * unsupported or invalid arguments. dtype YOCO_E4M3 sizes the scratch of
 * yoco_cross_attn_paged_e4m3.
 */
size_t yoco_cross_attn_workspace_size(int32_t max_rows, int32_t num_q_heads, int32_t num_kv_heads,
                                      int32_t head_dim, int32_t block_size, int32_t max_seq_len,
                                      yoco_dtype_t dtype);

/*
 * yoco_cross_attn_paged — one cross-decoder layer's causal paged GQA attention.
 *
 * "KV cache memory systems", "Cache contents": out = softmax(q K^T / sqrt(d_h)) V
 * over the cached keys up to the query position; "YOCO 论文与推理数据流详解"
 * §10.4 / §11: each of the L/2 cross-decoder layers queries the same shared
 * cache with its own Q, so this call runs once per layer over one cache.
 * Row i of the k_r rows of request r attends to seq_lens[r] - k_r + i + 1
 * keys (bottom-right causal, the query's own position included). Query head
 * h reads kv head h / (num_q_heads / num_kv_heads).
 *
 *   q, out                 device [max_rows][num_q_heads][head_dim], dtype; rows beyond
 *                          cross_query_start_loc[num_reqs] are neither read nor written
 *   k_cache, v_cache       device pools (layout above), dtype
 *   block_table, seq_lens  device int32, as for yoco_kv_append
 *   cross_query_start_loc  device int32 [num_reqs + 1] (from yoco_select_cross_rows)
 *   max_rows               host bound on the number of rows (grid size)
 *   max_seq_len            host bound on seq_lens (sizes the fp32 split-KV grid and its
 *                          workspace). A row with more keys sets YOCO_DEVERR_POS_RANGE; the
 *                          fp32 path then attends only to its first max_seq_len keys, so no
 *                          scratch beyond the workspace is ever touched (the bf16 path,
 *                          whose scratch does not depend on context length, attends to all
 *                          of them)
 *   scale                  softmax scale (1/sqrt(head_dim) for the pages' definition)
 *   flags                  bits of YOCO_ATTN_REVERSE | YOCO_ATTN_OVERLAP | YOCO_ATTN_KEEP_TAIL |
 *                          YOCO_ATTN_PLANNED (other bits are rejected; all are ignored on the
 *                          fp32 path).
 *                          PLANNED: the workspace holds the plan that yoco_cross_attn_plan made
 *                          for this step (same metadata arrays, unchanged since, and the same
 *                          max_rows, shapes and dtype), so the call launches the attention
 *                          kernel alone. Without it the call first makes that plan itself (one
 *                          more small kernel). A plan made for other shapes is detected: the
 *                          call then writes nothing and sets YOCO_DEVERR_PLAN.
 *                          REVERSE: the serial layers re-read one cache ("YOCO 论文与推理
 *                          数据流详解" §11); with the flag set on every other layer, a layer
 *                          starts on the pages the previous one read last, which are still
 *                          in L2. The result is the same up to summation order.
 *                          OVERLAP: the call is launched as a programmatic dependent of the
 *                          kernel before it on `stream`, so it reads block_table, seq_lens,
 *                          cross_query_start_loc, the cache and (with PLANNED) the plan while
 *                          that kernel drains. Set it only when that kernel writes none of
 *                          those (for example the previous cross-decoder layer, but not
 *                          yoco_cross_attn_plan); queries, outputs and the rest of the
 *                          workspace are touched only after that kernel has finished.
 *                          KEEP_TAIL: the pages are copied with an L2 evict-first hint except
 *                          the last ones each worker reads (evict-last, about 40 MB for a
 *                          bf16/fp32 cache, 20 MB for e4m3), which stay in L2 for the next
 *                          layer; meant for layers that alternate YOCO_ATTN_REVERSE over a
 *                          cache larger than L2. Hints only: the result is unchanged.
 *   workspace              device scratch of >= yoco_cross_attn_workspace_size(...) bytes,
 *                          16-byte aligned; contents need no initialisation (the plan is
 *                          written into it by yoco_cross_attn_plan or by a call without
 *                          PLANNED). One workspace serves one stream at a time.
 *   err_word               device int32 or NULL
 * Several cross rows of one request (max_rows > num_reqs: chunked prefill,
 * speculative verification) with at most 8 query heads per kv head are
 * walked together on the bf16 and e4m3 paths: consecutive rows of a request
 * share one pass over its pages (to the group's last row's causal end), each
 * row masked at its own end, so the cache is read once per group, not once
 * per row. A group holds 8 / G rows when ceil(max_rows / num_reqs) rows fit
 * in that (G <= 4), else 16 / G rows. Each row's result equals its own walk
 * up to summation order.
 * Long contexts are split across CTAs and merged with a log-sum-exp
 * combine in a fixed split order, so results do not depend on where pages
 * sit in the pool. Accuracy: fp32 accumulation; bf16 probabilities feed the
 * tensor-core P.V product.
 * The bf16 and e4m3 kernels run one CTA per SM, and the CTAs that share a
 * context cut between them wait (bounded) for each other before combining
 * it: every CTA of the grid must become resident. On a device whose SMs are
 * partitioned below its SM count (MPS thread limits, green contexts) such a
 * wait gives up after one second and sets YOCO_DEVERR_TIMEOUT.
 */
yoco_status_t yoco_cross_attn_paged(const void* q, const void* k_cache, const void* v_cache,
                                    void* out, const int32_t* block_table,
                                    int32_t max_blocks_per_req, const int32_t* seq_lens,
                                    const int32_t* cross_query_start_loc, int32_t num_reqs,
                                    int32_t max_rows, int32_t max_seq_len, int32_t num_q_heads,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                    int32_t num_blocks, float scale, yoco_dtype_t dtype,
                                    uint32_t flags, void* workspace, size_t workspace_bytes,
                                    int32_t* err_word, void* stream);

/*
 * yoco_cross_attn_plan — the per-step plan of the tensor-core attention.
 *
 * Every cross-decoder layer of a step attends with the same metadata to the
 * one shared cache ("YOCO 论文与推理数据流详解" §10.4, §11), so the way its
 * pages are dealt to the kernel's warps is the same for all of them. This
 * call works it out once, into `workspace`: each warp's first page and the
 * block-table entries of its first page copies, each CTA's first and last
 * segment, and the CTAs' arrival counters. The layers then pass
 * YOCO_ATTN_PLANNED and start streaming after one dependent load.
 *   arguments    as for yoco_cross_attn_paged (the same values the layers will pass);
 *                dtype YOCO_BF16 or YOCO_E4M3 (the e4m3 layers' own kernel shape);
 *                YOCO_F32 needs no plan and returns YOCO_OK without a launch
 *   flags        0 or YOCO_ATTN_OVERLAP (the previous kernel on `stream` writes none of
 *                block_table, seq_lens, cross_query_start_loc; the plan is written after it
 *                has finished)
 * Call it after the metadata of the step is final (after yoco_select_cross_rows), and again
 * whenever block_table, seq_lens, cross_query_start_loc or max_rows change.
 */
yoco_status_t yoco_cross_attn_plan(const int32_t* block_table, int32_t max_blocks_per_req,
                                   const int32_t* seq_lens, const int32_t* cross_query_start_loc,
                                   int32_t num_reqs, int32_t max_rows, int32_t max_seq_len,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t block_size, int32_t num_blocks, yoco_dtype_t dtype,
                                   uint32_t flags, void* workspace, size_t workspace_bytes,
                                   int32_t* err_word, void* stream);

/*
 * 8-bit cache: e4m3 K^/V^ with a K and a V scale per (page, kv head)
 * ---------------------------------------------------------------------
 * "KV cache memory systems", "Quantized cache changes attention inputs": a
 * quantized cache cuts the bytes per cached scalar and adds scale metadata;
 * keys and values may need separate calibration, per head. In YOCO the one
 * shared cache is what every cross-decoder layer streams ("YOCO 论文与推理
 * 数据流详解" §11, §18.2), so halving its bytes halves each layer's traffic;
 * one cache serves all layers, so there is no per-layer scale.
 *   - Pools hold one e4m3 byte per element (1 sign, 4 exponent bits with
 *     bias 7, 3 mantissa bits; largest finite 448; no infinities), in the
 *     layout above.
 *   - page_scales is device float32 [num_blocks][num_kv_heads][4]: the record
 *     of (page, kv head) is {k_scale, v_scale, unused, unused} (16 bytes, so
 *     one asynchronous copy fetches it with its page). Code c stands for
 *     value(c) * scale. The caller chooses the scales (calibration); a page
 *     keeps its scales while it holds tokens.
 *   - head_dim 128 or 256; block_size 16 or 32; groups up to 16 (as above).
 */

/*
 * yoco_kv_append_e4m3 — yoco_kv_append for an e4m3 cache: each element of
 * a new token's K^ (V^) row is stored as the e4m3 code nearest to
 * value / k_scale (value / v_scale) of its page and kv head, the division
 * in float32, ties to the even code, saturating at +-448.
 *   k_new, v_new   device bf16 [num_tokens][num_kv_heads][head_dim], 16-byte aligned
 *   k_cache, v_cache  device uint8 pools, 16-byte aligned
 *   page_scales    device float32 records (above), 16-byte aligned
 * A (token, kv head) whose page scale is not a positive finite number is
 * not written and sets YOCO_DEVERR_SCALE. Other arguments, checks and
 * device-side errors are those of yoco_kv_append.
 */
yoco_status_t yoco_kv_append_e4m3(const void* k_new, const void* v_new, void* k_cache,
                                  void* v_cache, const float* page_scales,
                                  const int32_t* block_table, int32_t max_blocks_per_req,
                                  const int32_t* seq_lens, const int32_t* query_start_loc,
                                  int32_t num_reqs, int32_t num_tokens, int32_t num_blocks,
                                  int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t* err_word, void* stream);

/*
 * yoco_cross_attn_paged_e4m3 — yoco_cross_attn_paged over an e4m3 cache.
 * Computes out = softmax(scale * q K^T) V with K = value(code) * k_scale and
 * V = value(code) * v_scale of each key's page and kv head.
 *   q, out        device bf16 [max_rows][num_q_heads][head_dim]
 *   k_cache, v_cache, page_scales  as for yoco_kv_append_e4m3
 *   workspace     >= yoco_cross_attn_workspace_size(..., YOCO_E4M3) bytes
 * Scales must lie in [2^-16, 2^7]; a page read with a scale outside that
 * range (or not finite) sets YOCO_DEVERR_SCALE and its result is undefined.
 * Arithmetic: codes widen exactly to f16, queries round to f16 (finite
 * queries must stay below 65504 in magnitude), f16 tensor-core products
 * with fp32 accumulation, f16 probabilities, and the V scale applied per
 * page in fp32. Everything else (flags, errors, determinism) is as for
 * yoco_cross_attn_paged.
 */
yoco_status_t yoco_cross_attn_paged_e4m3(const void* q, const void* k_cache, const void* v_cache,
                                         const float* page_scales, void* out,
                                         const int32_t* block_table, int32_t max_blocks_per_req,
                                         const int32_t* seq_lens,
                                         const int32_t* cross_query_start_loc, int32_t num_reqs,
                                         int32_t max_rows, int32_t max_seq_len,
                                         int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                         float scale, uint32_t flags, void* workspace,
                                         size_t workspace_bytes, int32_t* err_word, void* stream);

/*
 * yoco_cross_decode_step — a decode step's append and its first cross-decoder
 * layer in one launch (bf16 or e4m3 cache).
 *
 * For a decode-only batch (every request schedules exactly one new token and
 * gets one cross row, "You Only Cache Once, in vLLM", "Implementation in
 * vLLM"), this does what yoco_kv_append (or yoco_kv_append_e4m3) followed by
 * yoco_cross_attn_paged (or yoco_cross_attn_paged_e4m3) does for layer 0:
 * "YOCO 论文与推理数据流详解" §10.3–§10.4 — the token's K^/V^ is appended
 * once, and the layer's query attends to the keys up to and including it.
 * Later layers use yoco_cross_attn_paged(_e4m3) on the same cache.
 *   k_new, v_new      device bf16 [num_reqs][num_kv_heads][head_dim], 16-byte aligned
 *   query_start_loc   device int32 [num_reqs + 1] = 0, 1, ..., num_reqs (it is also the
 *                     cross query_start_loc); a request with another token count sets
 *                     YOCO_DEVERR_OFFSETS and its result is undefined
 *   seq_lens          tokens in the cache after this step (the new token included)
 *   dtype             YOCO_BF16 (page_scales ignored) or YOCO_E4M3 (page_scales as for
 *                     yoco_kv_append_e4m3); the pools hold that format
 *   workspace         >= yoco_cross_attn_workspace_size(num_reqs, ..., dtype) bytes
 * Other arguments, checks and errors are those of yoco_cross_attn_paged; of the flags
 * YOCO_ATTN_OVERLAP, YOCO_ATTN_KEEP_TAIL and YOCO_ATTN_PLANNED are taken (YOCO_ATTN_REVERSE
 * is rejected: the step walks its pages forward). Without PLANNED the call makes the
 * step's plan (query_start_loc as the cross query_start_loc), which the later layers of
 * the step can reuse with YOCO_ATTN_PLANNED. The cache ends bit-identical to the separate
 * append, and the output to the separate attention.
 */
yoco_status_t yoco_cross_decode_step(const void* q, const void* k_new, const void* v_new,
                                     void* k_cache, void* v_cache, const float* page_scales,
                                     void* out, const int32_t* block_table,
                                     int32_t max_blocks_per_req, const int32_t* seq_lens,
                                     const int32_t* query_start_loc, int32_t num_reqs,
                                     int32_t max_seq_len, int32_t num_q_heads,
                                     int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                     int32_t num_blocks, float scale, yoco_dtype_t dtype,
                                     uint32_t flags, void* workspace, size_t workspace_bytes,
                                     int32_t* err_word, void* stream);

/*
 * yoco_cross_attn_paged_noalloc — yoco_cross_attn_paged for callers that
 * cannot allocate device memory. The pages have no counterpart: this is a
 * library convenience, not part of the method.
 *
 * Some callers cannot call cudaMalloc: code running while a CUDA graph is
 * being captured, engines that carve out all device memory at start-up and
 * forbid later allocations, and plugin hosts that expose no allocator. This
 * entry point takes the same arguments as yoco_cross_attn_paged minus the
 * workspace, and keeps its scratch in one fixed array inside the library
 * (yoco_cross_attn_noalloc_capacity() bytes, 16 MiB), which every GPU that
 * loads the library holds until the process exits. It allocates nothing and
 * calls no allocating routine.
 *   - Returns YOCO_ERR_WORKSPACE, before any launch, when these bounds need
 *     more scratch than the array holds (yoco_cross_attn_workspace_size()
 *     gives the need).
 *   - dtype YOCO_F32 or YOCO_BF16 only: YOCO_E4M3 (and any other value)
 *     returns YOCO_ERR_UNSUPPORTED before any launch. No flags are taken:
 *     the call runs as yoco_cross_attn_paged with flags 0 (no REVERSE,
 *     OVERLAP, KEEP_TAIL or PLANNED), so each call makes its own plan in
 *     the array before its attention launch.
 *   - The first call on each device looks up the array's device address
 *     (with that device current); make that first call before any stream
 *     capture on the device. The address is kept for the life of the
 *     process: it assumes the device's primary context is never reset
 *     (no cudaDeviceReset between calls), since a reset reloads the module
 *     and moves the array.
 *   - Every call on a device shares the one array. The library writes each
 *     scratch word before reading it within a call, so no clearing is
 *     needed, but calls that overlap on the GPU (other streams, other host
 *     threads) race on it: serialise them.
 */
yoco_status_t yoco_cross_attn_paged_noalloc(const void* q, const void* k_cache,
                                            const void* v_cache, void* out,
                                            const int32_t* block_table,
                                            int32_t max_blocks_per_req, const int32_t* seq_lens,
                                            const int32_t* cross_query_start_loc,
                                            int32_t num_reqs, int32_t max_rows,
                                            int32_t max_seq_len, int32_t num_q_heads,
                                            int32_t num_kv_heads, int32_t head_dim,
                                            int32_t block_size, int32_t num_blocks, float scale,
                                            yoco_dtype_t dtype, int32_t* err_word, void* stream);

/* Bytes of the fixed scratch array used by yoco_cross_attn_paged_noalloc. */
size_t yoco_cross_attn_noalloc_capacity(void);

/*
 * yoco_set_l2_window — mark [base, base + bytes) as persisting in L2 for
 * work later enqueued on `stream` (bytes == 0 clears the window). The L2
 * set-aside is a property of this process's CUDA context only. Used to
 * keep a shared cache resident across the serial cross-decoder layers,
 * which re-read it one after another ("YOCO 论文与推理数据流详解" §11).
 * The window is cut to the device's largest window; hit_ratio in [0, 1]
 * is the fraction of its lines given the persisting property, and a
 * negative hit_ratio means "as many as the set-aside holds" (set-aside /
 * window), so that the same lines stay resident from one layer to the next.
 * Clearing the window (bytes == 0) also resets the lines already marked
 * persisting to normal (cudaCtxResetPersistingL2Cache) and the context's
 * persisting set-aside to zero, so that later kernels get the whole L2 back.
 */
yoco_status_t yoco_set_l2_window(void* stream, void* base, size_t bytes, float hit_ratio);

/*
 * yoco_cross_decoder_bytes — predicted HBM bytes of one scheduling step's
 * cross-decoder attention, for a traffic-aware scheduler. "YOCO 论文与推理数据流
 * 详解" §11 and §18.2: the global K^/V^ is written once but re-read by every
 * cross-decoder layer, so a request's decode traffic grows with its context
 * length times the number of cross-decoder layers. Per request r with k_r >= 1
 * cross rows (the yoco_select_cross_rows rule), whose last row attends to
 * kv = seq_lens[r] keys (clamped at 0); the rows share the request's pages,
 * which are read once:
 *   layers * ( kv * 2 * H_kv * head_dim * elem              K^ and V^
 *            + k_r * 2 * H_q * head_dim * elem              queries and outputs
 *            + 4 * ceil(kv / block_size) * H_kv )           block-table entries
 * with elem = 2 (bf16) or 4 (fp32); a request with no row moves nothing. For
 * one row per request this is each row's own causal prefix. For YOCO_E4M3 the
 * K^/V^ term uses 1 byte per element, the query/output term 2, and each page
 * adds its 16-byte scale record next to its block-table entry.
 *   query_start_loc, seq_lens   host int32 [num_reqs + 1] / [num_reqs]
 *   rows_per_req                host int32 [num_reqs] or NULL (= 1)
 *   per_req_bytes               host int64 out [num_reqs] or NULL
 * Returns the total, or -1 for invalid arguments. Pure host arithmetic.
 */
int64_t yoco_cross_decoder_bytes(const int32_t* query_start_loc, const int32_t* rows_per_req,
                                 const int32_t* seq_lens, int32_t num_reqs, int32_t layers,
                                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t block_size, yoco_dtype_t dtype, int64_t* per_req_bytes);

/*
 * yoco_selftest_wait_timeout — diagnostic for the bounded waits. The pages
 * have no counterpart. Launches one CTA that waits, with the library's
 * bounded-wait helper and a limit of limit_us microseconds (1..2000000), on
 * an asynchronous-copy barrier that nothing completes; the wait gives up,
 * the CTA sets YOCO_DEVERR_TIMEOUT in *err_word (device int32, required)
 * and returns, leaving the context usable. Used by the tests to show that a
 * copy that never lands ends in a status, not a hang.
 */
yoco_status_t yoco_selftest_wait_timeout(int32_t* err_word, uint32_t limit_us, void* stream);

/* Human-readable name of a status code (static string). */
const char* yoco_status_string(yoco_status_t status);

/*
 * The cudaError_t behind the most recent YOCO_ERR_CUDA returned on the
 * calling thread (0 if none yet), and its description (static string).
 */
int32_t yoco_last_cuda_error(void);
const char* yoco_last_cuda_error_string(void);

/* Library version as major * 10000 + minor * 100 + patch. */
int32_t yoco_version(void);

#ifdef __cplusplus
}
#endif

#endif /* YOCO_KV_H_ */
