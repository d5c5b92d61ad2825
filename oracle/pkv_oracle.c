/*
 * pkv_oracle.c -- plain, slow CPU oracle for the paged KV cache path of nano-vLLM.
 *
 * TEST INFRASTRUCTURE. Only the tests, the package smoke check and the benchmark's CPU
 * baseline (reference) leg may load this library. The CUDA library shares no code, header,
 * table or helper with it, and neither includes the other.
 *
 * Each function is the operation's definition written out, with no blocking, fusion or
 * reordering. Floating point is double precision: a bf16 input widens to double exactly,
 * every product and sum is taken in double, and every reduction runs in logical token
 * order, so a result does not depend on where a sequence's blocks sit in the pool.
 *
 * Sources (page title, section):
 *  [nano-vLLM 最小化vLLM重新实现] 架构 4 模型运行器: one KV tensor
 *      [2, num_layers, num_blocks, block_size, num_kv_heads, head_dim]; 架构 5 注意力机制:
 *      the store writes K/V into the paged cache through slot_mapping, prefill runs
 *      flash_attn_varlen_func (varlen, optional block_table for cached prefix blocks), decode
 *      runs flash_attn_with_kvcache over the paged cache; 关键设计选择: block size 256.
 *  [bxzpzcl.cn nano-vLLM 文章] §2.2.2 两级注意力加速: attention is
 *      softmax(q k^T / sqrt(head_dim)) v.
 *  [企业官网建设流程全解析 (Nano-vLLM 指南)] §2.2: each sequence keeps the list of its
 *      physical blocks like a page table; §4.4: prefix caching reuses the cached KV of a
 *      shared prefix and computes only the remaining tokens.
 *
 * Readings where the pages are silent (each is listed with its reason in the design notes):
 *  - slot = block_id * block_size + offset, a row of the [num_blocks * block_size,
 *    num_kv_heads, head_dim] view; a negative slot means "do not store" (padding token);
 *    slots of one call are unique.
 *  - query head hq reads KV head hq / (num_q_heads / num_kv_heads).
 *  - the scale is an argument (the pages use 1 / sqrt(head_dim)).
 *  - causal masking is aligned to the end of the keys: query i of a sequence with Lq queries
 *    and Lk keys sees keys j <= i + (Lk - Lq). With a cached prefix this is the only
 *    alignment under which the suffix rows equal the rows of the uncached computation.
 *  - a row with no visible key (context length 0) is all zeros.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_OK = 0, ORACLE_BAD_SLOT = 1, ORACLE_DUP_SLOT = 2, ORACLE_BAD_BLOCK = 3,
       ORACLE_BAD_ARG = 4, ORACLE_NO_MEMORY = 5, ORACLE_BAD_POSITION = 6 };

/* bf16 is the top half of an IEEE binary32; widening to double is exact. */
static double bf16_value(uint16_t bits)
{
    uint32_t word = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

/* Threads for one call: num_threads if positive, else every thread OpenMP offers. Passed to
 * each parallel region, so one call's choice does not carry over to the next call. */
static int threads_for(int32_t num_threads)
{
#ifdef _OPENMP
    return num_threads > 0 ? num_threads : omp_get_max_threads();
#else
    (void)num_threads;
    return 1;
#endif
}

int32_t pkv_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * store: k_cache[slot_mapping[t]] = k[t] and v_cache[slot_mapping[t]] = v[t] for each token t
 * with a non-negative slot. A row is num_kv_heads * head_dim bf16 words. k and v rows start
 * k_tok_stride / v_tok_stride words apart (they may be views into a fused qkv buffer).
 */
int32_t pkv_oracle_kv_store(const uint16_t *k, int64_t k_tok_stride,
                            const uint16_t *v, int64_t v_tok_stride,
                            const int64_t *slot_mapping, int64_t num_tokens,
                            uint16_t *k_cache, uint16_t *v_cache, int64_t num_slots,
                            int32_t num_kv_heads, int32_t head_dim)
{
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    if (num_tokens < 0 || num_slots < 0 || row <= 0) return ORACLE_BAD_ARG;
    unsigned char *seen = (unsigned char *)calloc((size_t)(num_slots > 0 ? num_slots : 1), 1);
    if (!seen) return ORACLE_NO_MEMORY;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_slots) { free(seen); return ORACLE_BAD_SLOT; }
        if (seen[slot]) { free(seen); return ORACLE_DUP_SLOT; }
        seen[slot] = 1;
    }
    free(seen);
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        for (int64_t e = 0; e < row; ++e) {
            k_cache[slot * row + e] = k[t * k_tok_stride + e];
            v_cache[slot * row + e] = v[t * v_tok_stride + e];
        }
    }
    return ORACLE_OK;
}

/*
 * One attention row: out[d] = sum_j p_j v_j[d] / sum_j p_j with p_j = exp(s_j - max s) and
 * s_j = scale * (q . k_j), over the n_keys keys whose rows are listed in key_rows (each an
 * offset, in bf16 words, of a key row for this head; the value row sits at the same offset
 * of v_base). score is caller scratch of n_keys doubles.
 */
static void attend_one(const uint16_t *q, const uint16_t *k_base, const uint16_t *v_base,
                       const int64_t *key_rows, int64_t n_keys, int32_t head_dim,
                       double scale, double *score, double *out)
{
    for (int32_t d = 0; d < head_dim; ++d) out[d] = 0.0;
    if (n_keys <= 0) return;
    for (int64_t j = 0; j < n_keys; ++j) {
        const uint16_t *kj = k_base + key_rows[j];
        double dot = 0.0;
        for (int32_t d = 0; d < head_dim; ++d) dot += bf16_value(q[d]) * bf16_value(kj[d]);
        score[j] = scale * dot;
    }
    double m = score[0];
    for (int64_t j = 1; j < n_keys; ++j)
        if (score[j] > m) m = score[j];
    double denom = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) {
        score[j] = exp(score[j] - m);
        denom += score[j];
    }
    for (int64_t j = 0; j < n_keys; ++j) {
        const uint16_t *vj = v_base + key_rows[j];
        for (int32_t d = 0; d < head_dim; ++d) out[d] += score[j] * bf16_value(vj[d]);
    }
    for (int32_t d = 0; d < head_dim; ++d) out[d] /= denom;
}

/*
 * Paged decode: for each sequence b and query head hq, one query q[b, hq, :] attends over the
 * first context_lens[b] logical tokens of the sequence. Logical token i lives in physical
 * block block_tables[b, i / block_size] at offset i % block_size of the per-layer pool
 * [num_blocks, block_size, num_kv_heads, head_dim]. out is [B, num_q_heads, head_dim].
 */
int32_t pkv_oracle_paged_decode(const uint16_t *q, const uint16_t *k_cache,
                                const uint16_t *v_cache, const int32_t *block_tables, int32_t W,
                                const int32_t *context_lens, int32_t B, int32_t num_q_heads,
                                int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                int64_t num_blocks, double scale, double *out,
                                int32_t num_threads)
{
    if (B < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_q_heads % num_kv_heads != 0)
        return ORACLE_BAD_ARG;
    const int32_t group = num_q_heads / num_kv_heads;
    int32_t status = ORACLE_OK;
    const int nthreads = threads_for(num_threads);
    (void)nthreads;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) num_threads(nthreads)
    for (int32_t b = 0; b < B; ++b) {
        for (int32_t hq = 0; hq < num_q_heads; ++hq) {
            const int32_t h = hq / group;
            const int64_t L = context_lens[b];
            double *o = out + ((int64_t)b * num_q_heads + hq) * head_dim;
            int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(L > 0 ? L : 1));
            double *score = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
            int ok = rows && score && L >= 0 && (L + block_size - 1) / block_size <= W;
            for (int64_t i = 0; ok && i < L; ++i) {
                const int64_t blk = block_tables[(int64_t)b * W + i / block_size];
                if (blk < 0 || blk >= num_blocks) { ok = 0; break; }
                const int64_t slot = blk * block_size + i % block_size;
                rows[i] = (slot * num_kv_heads + h) * head_dim;
            }
            if (ok) {
                attend_one(q + ((int64_t)b * num_q_heads + hq) * head_dim, k_cache, v_cache,
                           rows, L, head_dim, scale, score, o);
            } else {
                for (int32_t d = 0; d < head_dim; ++d) o[d] = NAN;
#pragma omp atomic write
                status = ORACLE_BAD_BLOCK;
            }
            free(rows);
            free(score);
        }
    }
    return status;
}

/*
 * Varlen prefill: sequence n has Lq = cu_seqlens_q[n+1] - cu_seqlens_q[n] queries (rows
 * cu_seqlens_q[n].. of q, [Tq, num_q_heads, head_dim] with token stride q_tok_stride) and
 * Lk = cu_seqlens_k[n+1] - cu_seqlens_k[n] keys. Query i attends over keys j <= i + (Lk - Lq)
 * when causal, over all Lk keys otherwise. Keys come from the packed k/v
 * ([Tk, num_kv_heads, head_dim], token stride kv_tok_stride, key j of sequence n at row
 * cu_seqlens_k[n] + j) or, when block_table is given, from the paged pools (key j at block
 * block_table[n, j / block_size], offset j % block_size; kv_tok_stride is then the pool's
 * row length num_kv_heads * head_dim). out is [Tq, num_q_heads, head_dim], densely packed.
 */
int32_t pkv_oracle_varlen_prefill(const uint16_t *q, int64_t q_tok_stride, const uint16_t *k,
                                  const uint16_t *v, int64_t kv_tok_stride,
                                  const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                  int32_t N, const int32_t *block_table, int32_t W,
                                  int32_t block_size, int64_t num_blocks, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, double scale,
                                  int32_t causal, double *out, int32_t num_threads)
{
    if (N < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        num_q_heads % num_kv_heads != 0 || (block_table && block_size <= 0))
        return ORACLE_BAD_ARG;
    const int32_t group = num_q_heads / num_kv_heads;
    int32_t status = ORACLE_OK;
    const int nthreads = threads_for(num_threads);
    (void)nthreads;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) num_threads(nthreads)
    for (int32_t n = 0; n < N; ++n) {
        for (int32_t hq = 0; hq < num_q_heads; ++hq) {
            const int32_t h = hq / group;
            const int64_t q0 = cu_seqlens_q[n], Lq = cu_seqlens_q[n + 1] - q0;
            const int64_t k0 = cu_seqlens_k[n], Lk = cu_seqlens_k[n + 1] - k0;
            int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(Lk > 0 ? Lk : 1));
            double *score = (double *)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
            int ok = rows && score && Lq >= 0 && Lk >= 0 &&
                     (!block_table || (Lk + block_size - 1) / block_size <= W);
            for (int64_t j = 0; ok && j < Lk; ++j) {
                int64_t key_row;
                if (block_table) {
                    const int64_t blk = block_table[(int64_t)n * W + j / block_size];
                    if (blk < 0 || blk >= num_blocks) { ok = 0; break; }
                    key_row = blk * block_size + j % block_size;
                } else {
                    key_row = k0 + j;
                }
                rows[j] = key_row * kv_tok_stride + (int64_t)h * head_dim;
            }
            for (int64_t i = 0; i < Lq; ++i) {
                double *o = out + ((q0 + i) * num_q_heads + hq) * head_dim;
                if (!ok) {
                    for (int32_t d = 0; d < head_dim; ++d) o[d] = NAN;
                    continue;
                }
                int64_t visible = causal ? i + (Lk - Lq) + 1 : Lk;
                if (visible > Lk) visible = Lk;
                attend_one(q + (q0 + i) * q_tok_stride + (int64_t)hq * head_dim, k, v, rows,
                           visible, head_dim, scale, score, o);
            }
            if (!ok) {
#pragma omp atomic write
                status = ORACLE_BAD_BLOCK;
            }
            free(rows);
            free(score);
        }
    }
    return status;
}

/*
 * QK normalisation and rotary position embedding of one layer's new tokens -- the step just
 * before the store. [nano-vLLM 最小化vLLM重新实现] 架构 6 模型: the Qwen3 layer applies an
 * RMSNorm to every query and key head (QK 归一化) and RoPE; 辅助层: RotaryEmbedding reads a
 * precomputed cos/sin cache.
 *
 * Token t's fused projection row (token stride tok_stride elements) holds num_q_heads query
 * heads, then num_kv_heads key heads, then num_kv_heads value heads, head_dim values each.
 * For a query or key head x with weight w (q_weight or k_weight, head_dim values):
 *     n_d = x_d / sqrt(mean_e(x_e^2) + eps) * w_d                              (RMSNorm)
 *     with half = head_dim / 2, c_i = cos_sin[pos, i], s_i = cos_sin[pos, half + i]:
 *     y_i        = n_i c_i - n_{i+half} s_i,   y_{i+half} = n_{i+half} c_i + n_i s_i
 * (the rotate-half pairing of element i with i + half). q_out [T, Hq, D] and k_out
 * [T, Hkv, D] get y; q_normed / k_normed get n (the test's error bound uses them). Value
 * heads pass through unchanged (the store copies them). A position outside
 * [0, max_position) is an error.
 */
int32_t pkv_oracle_qk_norm_rope(const uint16_t *qkv, int64_t tok_stride, int64_t num_tokens,
                                const int64_t *positions, const uint16_t *q_weight,
                                const uint16_t *k_weight, double eps, const float *cos_sin,
                                int64_t max_position, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_dim, double *q_out, double *k_out,
                                double *q_normed, double *k_normed)
{
    if (num_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        head_dim % 2 != 0 || tok_stride < (int64_t)(num_q_heads + 2 * num_kv_heads) * head_dim)
        return ORACLE_BAD_ARG;
    for (int64_t t = 0; t < num_tokens; ++t)
        if (positions[t] < 0 || positions[t] >= max_position) return ORACLE_BAD_POSITION;
    const int32_t half = head_dim / 2;
    const int32_t heads = num_q_heads + num_kv_heads;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < num_tokens; ++t) {
        const float *cs = cos_sin + positions[t] * head_dim;
        for (int32_t h = 0; h < heads; ++h) {
            const int is_q = h < num_q_heads;
            const uint16_t *x = qkv + t * tok_stride + (int64_t)h * head_dim;
            const uint16_t *w = is_q ? q_weight : k_weight;
            const int64_t orow = is_q ? (t * num_q_heads + h) * head_dim
                                      : (t * num_kv_heads + (h - num_q_heads)) * head_dim;
            double *n = (is_q ? q_normed : k_normed) + orow;
            double *y = (is_q ? q_out : k_out) + orow;
            double ss = 0.0;
            for (int32_t d = 0; d < head_dim; ++d) ss += bf16_value(x[d]) * bf16_value(x[d]);
            const double r = 1.0 / sqrt(ss / head_dim + eps);
            for (int32_t d = 0; d < head_dim; ++d) n[d] = bf16_value(x[d]) * r * bf16_value(w[d]);
            for (int32_t i = 0; i < half; ++i) {
                const double c = cs[i], sn = cs[half + i];
                y[i] = n[i] * c - n[i + half] * sn;
                y[i + half] = n[i + half] * c + n[i] * sn;
            }
        }
    }
    return ORACLE_OK;
}
