/*
 * CPU oracle for the YOCO cross-decoder hot path — TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct restatements of what the three library
 * calls compute. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load this file's library. It shares no code, header,
 * table or helper with the CUDA library: it is written from the pages'
 * definitions alone.
 *
 *   append    — "YOCO 论文与推理数据流详解" §10.3 (each new token's shared
 *               K^/V^ is appended once to the one global cache) and §7.3;
 *               "KV cache memory systems", "Contiguous allocation wastes
 *               capacity" (a block table maps logical token blocks to
 *               physical pages). Layout reading: pools are
 *               [num_blocks][H_kv][block_size][D]; token position p of a
 *               request lives in page block_table[p / block_size] at slot
 *               p % block_size.
 *   select    — "You Only Cache Once, in vLLM", "Implementation in vLLM":
 *               every request collapses to its last scheduled token(s) for
 *               the cross-decoder; the fast-prefill metadata builder gives
 *               each request k_r rows, a new query_start_loc that is the
 *               running sum of k_r, and keeps seq_lens unchanged.
 *   attention — "KV cache memory systems", "Cache contents":
 *               out = softmax(q K^T / sqrt(d_h)) V over the keys at or before
 *               the query position; "YOCO 论文与推理数据流详解" §10.4: every
 *               cross-decoder layer queries the same K^/V^ with its own Q.
 *               GQA reading: query head h uses kv head h / (H_q / H_kv).
 *               Causal reading (bottom-right, inclusive): row i of the k_r
 *               rows of a request with seq_len tokens sees
 *               seq_len - k_r + i + 1 keys.
 *
 *   e4m3      — "KV cache memory systems", "Quantized cache changes attention
 *               inputs": the cache may hold 8-bit values plus per-page,
 *               per-head K and V scales (see the e4m3 section below).
 *
 * Arithmetic is float64 throughout, except where a float32 division decides
 * an 8-bit code; bf16 inputs arrive already widened exactly to double by the
 * caller.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ select */

/*
 * rows_per_req may be NULL (one row per request). A request with q_len
 * scheduled tokens contributes k = min(want, q_len) rows: its last k token
 * indices, in order. Returns the number of rows, or -1 if some q_len or
 * want is negative (the output is then not meaningful).
 */
int64_t oracle_select_cross_rows(const int32_t* qsl, const int32_t* rows_per_req,
                                 int32_t num_reqs, int32_t* rows, int32_t* cqsl)
{
    int64_t n = 0;
    int bad = 0;
    cqsl[0] = 0;
    for (int32_t r = 0; r < num_reqs; ++r) {
        int64_t q_len = (int64_t)qsl[r + 1] - (int64_t)qsl[r];
        int64_t want = rows_per_req ? rows_per_req[r] : 1;
        if (q_len < 0 || want < 0) {
            bad = 1;
            q_len = 0;
            want = 0;
        }
        int64_t k = want < q_len ? want : q_len;
        for (int64_t i = 0; i < k; ++i) {
            rows[n] = (int32_t)(qsl[r + 1] - k + i);
            ++n;
        }
        cqsl[r + 1] = (int32_t)n;
    }
    return bad ? -1 : n;
}

/* ------------------------------------------------------------------ append */

/*
 * Writes k_new/v_new ([T][H_kv][D], elem_bytes each) into the pools.
 * Token j of request r (j < q_len) sits at position seq_lens[r] - q_len + j.
 * Tokens whose position or page is out of range are skipped and counted;
 * the return value is that count (0 = every token written).
 */
int64_t oracle_kv_append(const uint8_t* k_new, const uint8_t* v_new, uint8_t* k_pool,
                         uint8_t* v_pool, const int32_t* block_table, int32_t max_blocks,
                         const int32_t* seq_lens, const int32_t* qsl, int32_t num_reqs,
                         int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                         int32_t head_dim, int32_t elem_bytes)
{
    int64_t skipped = 0;
    const size_t row = (size_t)head_dim * (size_t)elem_bytes;
    for (int32_t r = 0; r < num_reqs; ++r) {
        int64_t q_len = (int64_t)qsl[r + 1] - (int64_t)qsl[r];
        for (int64_t j = 0; j < q_len; ++j) {
            int64_t tok = (int64_t)qsl[r] + j;
            int64_t pos = (int64_t)seq_lens[r] - q_len + j;
            if (pos < 0 || pos / block_size >= max_blocks) {
                skipped += num_kv_heads;
                continue;
            }
            int64_t page = block_table[(int64_t)r * max_blocks + pos / block_size];
            int64_t slot = pos % block_size;
            if (page < 0 || page >= num_blocks) {
                skipped += num_kv_heads;
                continue;
            }
            for (int32_t h = 0; h < num_kv_heads; ++h) {
                size_t dst = (size_t)(((page * num_kv_heads + h) * block_size + slot)) * row;
                size_t src = (size_t)(tok * num_kv_heads + h) * row;
                memcpy(k_pool + dst, k_new + src, row);
                memcpy(v_pool + dst, v_new + src, row);
            }
        }
    }
    return skipped;
}

/* -------------------------------------------------------------- e4m3 cache */

/*
 * "KV cache memory systems", "Quantized cache changes attention inputs": a
 * quantized cache stores fewer bytes per scalar and adds scale metadata;
 * keys and values may need separate calibration, per head. Readings: the
 * 8-bit format is e4m3 (sign bit, 4 exponent bits with bias 7, 3 mantissa
 * bits, subnormals, no infinities, S.1111.111 = NaN, largest finite 448);
 * each (physical page, kv head) has one scale for K and one for V, given by
 * the caller as a record of four floats {k_scale, v_scale, unused, unused};
 * code c stands for decode(c) * scale, and a value x is stored as
 * encode(x / scale), the division in float32, rounded to the nearest code
 * with ties to the even code, saturating at +-448.
 */
double oracle_e4m3_decode(uint8_t c)
{
    int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);        /* (m / 8) * 2^-6 */
    else
        v = ldexp(8.0 + m, e - 10);      /* (1 + m / 8) * 2^(e - 7) */
    return sign ? -v : v;
}

uint8_t oracle_e4m3_encode(float x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7E;
    int code;
    if (a < ldexp(1.0, -6)) {
        /* subnormal spacing 2^-9; a result of 8 is the smallest normal */
        code = (int)nearbyint(ldexp(a, 9));
    } else {
        int e2;
        frexp(a, &e2);                   /* a in [2^(e2-1), 2^e2) */
        int e = e2 - 1;
        int M = (int)nearbyint(ldexp(a, 3 - e));  /* 8..16; 16 carries into the exponent */
        code = ((e + 7) << 3) + (M - 8);
    }
    if (code > 0x7E)
        code = 0x7E;
    return sign | (uint8_t)code;
}

void oracle_e4m3_encode_array(const float* x, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_encode(x[i]);
}

void oracle_e4m3_decode_array(const uint8_t* c, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_decode(c[i]);
}

static float bf16_bits_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * Append with quantisation: k_new/v_new are bf16 bits [T][H_kv][D]; pools
 * hold one e4m3 byte per element, [num_blocks][H_kv][block_size][D];
 * scales is [num_blocks][H_kv][4] floats. Placement is the one of
 * oracle_kv_append. A (token, head) whose scale is not a positive finite
 * number is skipped; skipped (token, head) pairs are counted and returned.
 */
int64_t oracle_kv_append_e4m3(const uint16_t* k_new, const uint16_t* v_new, uint8_t* k_pool,
                              uint8_t* v_pool, const float* scales, const int32_t* block_table,
                              int32_t max_blocks, const int32_t* seq_lens, const int32_t* qsl,
                              int32_t num_reqs, int32_t num_blocks, int32_t block_size,
                              int32_t num_kv_heads, int32_t head_dim)
{
    int64_t skipped = 0;
    for (int32_t r = 0; r < num_reqs; ++r) {
        int64_t q_len = (int64_t)qsl[r + 1] - (int64_t)qsl[r];
        for (int64_t j = 0; j < q_len; ++j) {
            int64_t tok = (int64_t)qsl[r] + j;
            int64_t pos = (int64_t)seq_lens[r] - q_len + j;
            if (pos < 0 || pos / block_size >= max_blocks) {
                skipped += num_kv_heads;
                continue;
            }
            int64_t page = block_table[(int64_t)r * max_blocks + pos / block_size];
            int64_t slot = pos % block_size;
            if (page < 0 || page >= num_blocks) {
                skipped += num_kv_heads;
                continue;
            }
            for (int32_t h = 0; h < num_kv_heads; ++h) {
                const float ks = scales[(page * num_kv_heads + h) * 4 + 0];
                const float vs = scales[(page * num_kv_heads + h) * 4 + 1];
                if (!(ks > 0.0f) || !(vs > 0.0f) || isinf(ks) || isinf(vs)) {
                    ++skipped;
                    continue;
                }
                size_t dst = (size_t)((page * num_kv_heads + h) * block_size + slot) * head_dim;
                size_t src = (size_t)(tok * num_kv_heads + h) * head_dim;
                for (int32_t d = 0; d < head_dim; ++d) {
                    const float kq = bf16_bits_to_float(k_new[src + d]) / ks;
                    const float vq = bf16_bits_to_float(v_new[src + d]) / vs;
                    k_pool[dst + d] = oracle_e4m3_encode(kq);
                    v_pool[dst + d] = oracle_e4m3_encode(vq);
                }
            }
        }
    }
    return skipped;
}

/*
 * The first n_tokens positions of one request read back through its block
 * table row and dequantised: out[pos][h][d] = decode(code) * scale, with
 * scale = scales[page][h][which] (which = 0 for K, 1 for V). Returns 0, or
 * -1 if a page index is out of range (those entries are left untouched).
 */
int32_t oracle_e4m3_gather(const uint8_t* pool, const float* scales, int32_t which,
                           const int32_t* bt_row, int64_t n_tokens, int32_t num_blocks,
                           int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                           double* out)
{
    int32_t st = 0;
    for (int64_t pos = 0; pos < n_tokens; ++pos) {
        int64_t page = bt_row[pos / block_size], slot = pos % block_size;
        if (page < 0 || page >= num_blocks) {
            st = -1;
            continue;
        }
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            const double sc = (double)scales[(page * num_kv_heads + h) * 4 + which];
            const uint8_t* src = pool + ((page * num_kv_heads + h) * block_size + slot) * head_dim;
            double* dst = out + (pos * num_kv_heads + h) * head_dim;
            for (int32_t d = 0; d < head_dim; ++d)
                dst[d] = oracle_e4m3_decode(src[d]) * sc;
        }
    }
    return st;
}

/* --------------------------------------------------------------- attention */

/*
 * One query row against one request's contiguous keys/values.
 *   q   [H_q][D], K/V [kv_len][H_kv][D] (only the first kv_len are read),
 *   out [H_q][D], w: scratch of kv_len doubles.
 */
void oracle_attn_row(const double* q, const double* K, const double* V, int64_t kv_len,
                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, double scale,
                     double* out, double* w)
{
    const int32_t group = num_q_heads / num_kv_heads;
    for (int32_t h = 0; h < num_q_heads; ++h) {
        const int32_t g = h / group;
        const double* qh = q + (int64_t)h * head_dim;
        double m = -INFINITY;
        for (int64_t t = 0; t < kv_len; ++t) {
            const double* kt = K + (t * num_kv_heads + g) * head_dim;
            double s = 0.0;
            for (int32_t d = 0; d < head_dim; ++d) s += qh[d] * kt[d];
            w[t] = scale * s;
            if (w[t] > m) m = w[t];
        }
        double denom = 0.0;
        for (int64_t t = 0; t < kv_len; ++t) {
            w[t] = exp(w[t] - m);
            denom += w[t];
        }
        double* oh = out + (int64_t)h * head_dim;
        for (int32_t d = 0; d < head_dim; ++d) {
            double acc = 0.0;
            for (int64_t t = 0; t < kv_len; ++t) acc += w[t] * V[(t * num_kv_heads + g) * head_dim + d];
            oh[d] = acc / denom;
        }
    }
}

typedef struct {
    const double* q;
    const double* const* K_req;
    const double* const* V_req;
    const int32_t* seq_lens;
    const int32_t* cqsl;
    const int32_t* row_list; /* rows to compute (indices into the row axis) */
    int64_t n_list;
    int32_t num_reqs, num_q_heads, num_kv_heads, head_dim;
    double scale;
    double* out;
    const int64_t* cap;      /* rows available in K_req[r] / V_req[r] */
    int64_t max_len;
    int64_t next;            /* next index of row_list to take */
    pthread_mutex_t mu;
    int bad;
} attn_job_t;

static int32_t request_of_row(const int32_t* cqsl, int32_t num_reqs, int64_t n)
{
    for (int32_t r = 0; r < num_reqs; ++r)
        if (n < cqsl[r + 1]) return r;
    return -1;
}

static void* attn_worker(void* arg)
{
    attn_job_t* J = (attn_job_t*)arg;
    double* w = (double*)malloc(sizeof(double) * (size_t)(J->max_len > 0 ? J->max_len : 1));
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int64_t i = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (i >= J->n_list) break;
        int64_t n = J->row_list[i];
        double* o = J->out + i * (int64_t)J->num_q_heads * J->head_dim;
        int32_t r = request_of_row(J->cqsl, J->num_reqs, n);
        int64_t kv_len = -1;
        if (r >= 0) {
            int64_t k = (int64_t)J->cqsl[r + 1] - J->cqsl[r];
            kv_len = (int64_t)J->seq_lens[r] - k + (n - J->cqsl[r]) + 1;
        }
        if (r < 0 || kv_len <= 0 || kv_len > J->cap[r]) {
            memset(o, 0, sizeof(double) * (size_t)J->num_q_heads * J->head_dim);
            pthread_mutex_lock(&J->mu);
            J->bad = 1;
            pthread_mutex_unlock(&J->mu);
            continue;
        }
        oracle_attn_row(J->q + n * (int64_t)J->num_q_heads * J->head_dim, J->K_req[r], J->V_req[r],
                        kv_len, J->num_q_heads, J->num_kv_heads, J->head_dim, J->scale, o, w);
    }
    free(w);
    return NULL;
}

/*
 * Cross-decoder attention for the rows listed in row_list (n_list of them).
 *   q        [num_rows][H_q][D]   (row axis as produced by select)
 *   K_req[r], V_req[r]            contiguous [len_r][H_kv][D], len_r >= seq_lens[r]
 *   cqsl     [num_reqs + 1]       cross query_start_loc from select
 *   out      [n_list][H_q][D]     out[i] belongs to row row_list[i]
 *   cap[r]   rows held by K_req[r] / V_req[r]; every kv_len must fit
 * Returns 0, or -1 when some listed row has no request or a non-positive /
 * over-long key count (its output is zero-filled).
 */
int32_t oracle_cross_attn(const double* q, const double* const* K_req, const double* const* V_req,
                          const int32_t* seq_lens, const int32_t* cqsl, int32_t num_reqs,
                          const int32_t* row_list, int64_t n_list, int32_t num_q_heads,
                          int32_t num_kv_heads, int32_t head_dim, double scale, double* out,
                          const int64_t* cap, int32_t nthreads)
{
    attn_job_t J;
    J.q = q; J.K_req = K_req; J.V_req = V_req; J.seq_lens = seq_lens; J.cqsl = cqsl;
    J.row_list = row_list; J.n_list = n_list; J.num_reqs = num_reqs;
    J.num_q_heads = num_q_heads; J.num_kv_heads = num_kv_heads; J.head_dim = head_dim;
    J.scale = scale; J.out = out; J.cap = cap; J.next = 0; J.bad = 0;
    J.max_len = 1;
    for (int32_t r = 0; r < num_reqs; ++r)
        if (cap[r] > J.max_len) J.max_len = cap[r];
    pthread_mutex_init(&J.mu, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads == 1) {
        attn_worker(&J);
    } else {
        pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
        for (int32_t i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, attn_worker, &J);
        for (int32_t i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&J.mu);
    return J.bad ? -1 : 0;
}
