/*
 * pkv.h -- C ABI of libpkv, the paged KV cache kernels for GB300 (sm_103a).
 *
 * The library implements the data-parallel hot path of the paged KV cache that the nano-vLLM
 * pages describe («nano-vLLM 最小化vLLM重新实现», 架构 4 模型运行器 and 架构 5 注意力机制):
 *
 *   pkv_kv_store             store each new token's K/V into the block pool via slot_mapping
 *   pkv_paged_decode_attn    one query token per sequence over its paged KV (GQA)
 *   pkv_varlen_prefill_attn  causal attention over cu_seqlens-packed prompts, keys either
 *                            packed or read from the pool through a block table
 *
 * Common rules
 *  - Every pointer argument except `stream` is a DEVICE pointer, allocated and owned by the
 *    caller. The library allocates nothing and frees nothing; it keeps no pointer after a
 *    call returns.
 *  - bf16 tensors are passed as `void*` to 16-bit storage. The innermost dimension (head_dim)
 *    is contiguous; token strides are given in elements where the argument list has one.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Every call only enqueues
 *    work on it: it never synchronises the host, so it may be captured into a CUDA graph.
 *  - The KV pool of one layer is [num_blocks, block_size, num_kv_heads, head_dim] bf16, i.e.
 *    one slice of the engine's [2, num_layers, num_blocks, block_size, num_kv_heads,
 *    head_dim] tensor; K and V pools are separate pointers with the same layout. A "slot" is
 *    block_id * block_size + offset, a row of the [num_blocks * block_size, num_kv_heads,
 *    head_dim] view.
 *  - Errors in scalar arguments are found on the host before anything is enqueued and are
 *    returned as a status; nothing is written then. Shapes that are valid but that the
 *    kernels do not implement return PKV_ERR_UNSUPPORTED. A failed launch returns
 *    PKV_ERR_CUDA. Zero-size work (no tokens, no sequences) returns PKV_OK and enqueues
 *    nothing.
 *  - Errors in device DATA (a slot or block id out of range, a context longer than the
 *    block table row) cannot be seen by the host without a sync. The kernels skip the bad
 *    access (no out-of-bounds read or write happens) and set a bit in a device-side error
 *    word, which pkv_get_device_errors() reads.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t pkv_status;

#define PKV_OK 0
#define PKV_ERR_INVALID_ARG 1 /* null pointer, negative size, Hq % Hkv != 0, bad stride */
#define PKV_ERR_UNSUPPORTED 2 /* valid but not implemented: head_dim != 128, block_size % 256 */
#define PKV_ERR_WORKSPACE 3   /* workspace missing or smaller than the query says */
#define PKV_ERR_CUDA 4        /* a CUDA runtime/driver call failed (launch, tensor map) */
#define PKV_ERR_NO_BLOCKS 5   /* block manager: not enough free blocks; nothing was changed */

/* bits of the device-side error word */
#define PKV_DEVERR_SLOT_RANGE 1u      /* kv_store: slot_mapping[t] >= num_slots */
#define PKV_DEVERR_BLOCK_RANGE 2u     /* attention: block id < 0 or >= num_blocks */
#define PKV_DEVERR_CONTEXT_RANGE 4u   /* decode: context_lens[b] < 0, > max_context_len,
                                         or > block_table_width * block_size */
#define PKV_DEVERR_SEQLEN_RANGE 8u    /* prefill: bad cu_seqlens entry */
#define PKV_DEVERR_POSITION_RANGE 32u /* qk_norm_rope_store: position outside the cos/sin
                                         cache */
#define PKV_DEVERR_TIMEOUT 16u        /* a pipeline wait gave up after 2 s. The bit is sticky:
                                         while it is set, every attention kernel of the library
                                         returns at once without computing, until
                                         pkv_get_device_errors(&e, 1) clears it. */
#define PKV_DEVERR_WORKSPACE 64u      /* decode: the work counter at the start of the workspace
                                         held a value that a zeroed counter cannot give: it
                                         was not zero when the call started, and outputs may
                                         be missing. Zero it again (cudaMemsetAsync). */

/* Human-readable name of a status code. Never NULL; the string is static. */
const char *pkv_status_string(pkv_status status);

/* Version of this ABI (incremented on any incompatible change). */
int32_t pkv_abi_version(void);

/*
 * Read the device-side error word of the current device (the OR of the PKV_DEVERR_* bits set
 * by kernels since the last reset) into *errors, and reset it to 0 when `reset` != 0.
 * Synchronises the current device first: a diagnostic, not for the hot loop.
 */
pkv_status pkv_get_device_errors(uint32_t *errors, int32_t reset);

/*
 * OR `bits` (PKV_DEVERR_* values) into the device-side error word of the current device.
 * Setting PKV_DEVERR_TIMEOUT makes every later kernel of the library return without
 * computing, exactly as after a wait that gave up; this is how the abort path is exercised
 * without stalling anything. Synchronises the current device first. Returns
 * PKV_ERR_CUDA if the device cannot be reached.
 */
pkv_status pkv_raise_device_errors(uint32_t bits);

/*
 * kv_store -- the Triton store_kvcache of nano-vLLM («nano-vLLM 最小化vLLM重新实现»,
 * 架构 5: "writes K/V into the paged cache using slot_mapping, no Python loop").
 *
 * For every token t in [0, num_tokens) with slot_mapping[t] >= 0:
 *     k_cache[slot_mapping[t], :, :] = k[t, :, :]
 *     v_cache[slot_mapping[t], :, :] = v[t, :, :]
 * A negative slot skips the token (padding). Slots of one call must be unique (a duplicate
 * leaves one of the two rows, which one is unspecified). A slot >= num_slots is skipped and
 * sets PKV_DEVERR_SLOT_RANGE.
 *
 * k, v:          [num_tokens, num_kv_heads, head_dim] bf16; token t's row starts
 *                k_tok_stride (v_tok_stride) elements after token t-1's, and a row's
 *                num_kv_heads * head_dim elements are contiguous (views into a fused qkv
 *                buffer are fine). Strides must be >= num_kv_heads * head_dim.
 * slot_mapping:  [num_tokens] int64.
 * k_cache, v_cache: [num_slots, num_kv_heads, head_dim] bf16 (a per-layer pool,
 *                num_slots = num_blocks * block_size).
 * Returns PKV_ERR_INVALID_ARG for null pointers with num_tokens > 0, negative sizes, or
 * strides shorter than a row. Any head count and head_dim are accepted: rows whose byte
 * length, strides and addresses are multiples of 16 bytes move with bulk copies through
 * shared memory (16-byte vectors for rows over 48 KiB), other rows two bytes at a time.
 */
pkv_status pkv_kv_store(const void *k, int64_t k_tok_stride, const void *v, int64_t v_tok_stride,
                        const int64_t *slot_mapping, int64_t num_tokens, void *k_cache,
                        void *v_cache, int64_t num_slots, int32_t num_kv_heads,
                        int32_t head_dim, void *stream);

/*
 * Bytes of device workspace that pkv_paged_decode_attn needs for these sizes (at least 16).
 * `num_splits` must be the value later passed to the call (0 = automatic choice, made from
 * the sizes and the current device's SM count). The workspace holds each split's partial
 * output [batch, num_q_heads, splits, head_dim] fp32 and its log-sum-exp [batch,
 * num_q_heads, splits] fp32 (when there is more than one split), after a 16-byte header
 * that holds the persistent kernel's work counter (see the workspace argument below: it must
 * be zero before the first call). Returns 0 for invalid sizes.
 */
size_t pkv_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_context_len,
                                  int32_t num_splits);

/*
 * paged_decode_attn -- flash_attn_with_kvcache over the paged cache («nano-vLLM
 * 最小化vLLM重新实现», 架构 5: decode uses the paged KV cache through block tables and
 * cache lengths), written as split-K flash-decoding.
 *
 * For each sequence b in [0, batch) and query head hq in [0, num_q_heads), with
 * h = hq / (num_q_heads / num_kv_heads) and L = context_lens[b]:
 *     key/value i (0 <= i < L) is row  block_tables[b, i / block_size] * block_size
 *                                       + i % block_size  of k_cache / v_cache, head h
 *     s_i = scale * dot(q[b, hq, :], k_i)
 *     out[b, hq, :] = sum_i exp(s_i - max s) v_i / sum_i exp(s_i - max s)    (bf16, RNE)
 * L = 0 gives zeros. The token stored this step is expected at position L - 1, so the call
 * comes after pkv_kv_store on the same stream.
 *
 * q:             [batch, num_q_heads, head_dim] bf16, contiguous.
 * k_cache, v_cache: [num_blocks, block_size, num_kv_heads, head_dim] bf16.
 * block_tables:  [batch, block_table_width] int32; only the first ceil(L / block_size)
 *                entries of row b are read (padding entries are never dereferenced).
 * context_lens:  [batch] int32, each <= max_context_len.
 * num_splits:    0 = automatic; otherwise the number of KV splits for the longest context
 *                (each split covers the same number of logical tokens, a multiple of 64;
 *                shorter sequences use fewer splits). Results are identical for any
 *                physical placement of the blocks; they differ by rounding across values of
 *                num_splits.
 * workspace:     pkv_decode_workspace_bytes(...) bytes, 16-byte aligned, private to this
 *                call while it runs (calls that may overlap need separate workspaces). Its
 *                first 4 bytes are the persistent kernel's work counter: it must be zero
 *                before the workspace's first call (e.g. cudaMemsetAsync of the first 16
 *                bytes once after allocating it), and every call leaves it at zero again,
 *                so calls on the same stream need nothing in between, also in a captured
 *                CUDA graph. With a counter that was not zero the results are undefined
 *                (never a fault); values that a zeroed counter cannot give set
 *                PKV_DEVERR_WORKSPACE. The rest of the workspace is scratch.
 * out:           [batch, num_q_heads, head_dim] bf16.
 * Implemented: head_dim == 128, block_size a multiple of 256 (the pages: block size must be
 * a multiple of 256), any num_q_heads / num_kv_heads, q, pools and out 16-byte aligned.
 */
pkv_status pkv_paged_decode_attn(const void *q, const void *k_cache, const void *v_cache,
                                 const int32_t *block_tables, int32_t block_table_width,
                                 const int32_t *context_lens, int32_t batch,
                                 int32_t max_context_len, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                 int64_t num_blocks, float scale, int32_t num_splits,
                                 void *workspace, size_t workspace_bytes, void *out,
                                 void *stream);

/*
 * paged_decode_step -- one decode step of a layer in one call: each sequence's new token is
 * written into the pools at slot_mapping[b] (as pkv_kv_store does: «nano-vLLM 最小化vLLM重新实现»,
 * 架构 5, the store through slot_mapping) and then every sequence attends over its context
 * (as pkv_paged_decode_attn, whose arguments and workspace these are). The store happens
 * inside the decode kernel: the part of the kernel that reads a sequence's last position for
 * a KV head writes that row first, so the step needs no separate store kernel (with more than
 * one CTA per KV head -- num_q_heads / num_kv_heads >= 3 -- a store kernel runs first instead).
 *
 * k_new, v_new: [batch, num_kv_heads, head_dim] bf16, token strides in elements (multiples of
 *               8); slot_mapping: [batch] int64. The new token of sequence b is position
 *               context_lens[b] - 1 and slot_mapping[b] must be that position's slot in b's
 *               block table; a negative slot stores nothing (a padding row). A sequence with
 *               context length 0 stores nothing. A slot may not be read by another sequence
 *               in the same call (new tokens go to a sequence's own blocks). Slot >=
 *               num_blocks * block_size: skipped, PKV_DEVERR_SLOT_RANGE.
 * The result equals pkv_kv_store followed by pkv_paged_decode_attn, bit for bit.
 */
pkv_status pkv_paged_decode_step(const void *q, const void *k_new, int64_t k_new_tok_stride,
                                 const void *v_new, int64_t v_new_tok_stride,
                                 const int64_t *slot_mapping, void *k_cache, void *v_cache,
                                 const int32_t *block_tables, int32_t block_table_width,
                                 const int32_t *context_lens, int32_t batch,
                                 int32_t max_context_len, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                 int64_t num_blocks, float scale, int32_t num_splits,
                                 void *workspace, size_t workspace_bytes, void *out,
                                 void *stream);

/*
 * Bytes of device workspace that pkv_varlen_prefill_attn needs for num_seqs sequences of at
 * most max_seqlen_q queries: a 16-byte header (the persistent kernel's work counter and the
 * length of its work list), about 12 bytes per sequence and 8 per possible query-block count
 * for sorting, and the work list itself, 8 bytes per (sequence, 128-query block):
 * about 16 + 12 * num_seqs + 8 * num_seqs * ceil(max_seqlen_q / 128). The call writes all of
 * it on its stream before the attention kernel runs, so its contents need no initialisation.
 * Returns 0 for invalid sizes, or when the list would exceed 2^31 - 1 entries.
 */
size_t pkv_prefill_workspace_bytes(int32_t num_seqs, int32_t max_seqlen_q,
                                   int32_t num_q_heads, int32_t head_dim);

/*
 * varlen_prefill_attn -- flash_attn_varlen_func («nano-vLLM 最小化vLLM重新实现», 架构 5:
 * prefill over variable-length sequences, with an optional block_table for prefix caching).
 *
 * Sequence n has Lq = cu_seqlens_q[n+1] - cu_seqlens_q[n] queries and
 * Lk = cu_seqlens_k[n+1] - cu_seqlens_k[n] keys. For query i of sequence n and query head hq
 * (KV head h = hq / (num_q_heads / num_kv_heads)):
 *     visible keys  j <= i + (Lk - Lq)  when causal != 0 (aligned to the end of the keys, so
 *                   with a cached prefix query i sits at absolute position Lk - Lq + i),
 *                   all Lk keys otherwise
 *     out[cu_seqlens_q[n] + i, hq, :] = softmax_j(scale * q . k_j) v_j          (bf16, RNE)
 * A query that sees no key (Lq > Lk with causal) gets zeros.
 *
 * q:             [total_q, num_q_heads, head_dim] bf16, token stride q_tok_stride elements;
 *                total_q >= cu_seqlens_q[num_seqs] (the rows the tensor really has: tiles
 *                that reach past them read zeros instead).
 * k, v:          block_table == NULL: packed [total_k, num_kv_heads, head_dim] bf16, key j of
 *                sequence n at row cu_seqlens_k[n] + j, token stride kv_tok_stride;
 *                total_k >= cu_seqlens_k[num_seqs].
 *                block_table != NULL: the per-layer pools [num_blocks, block_size,
 *                num_kv_heads, head_dim]; key j of sequence n at row
 *                block_table[n, j / block_size] * block_size + j % block_size;
 *                kv_tok_stride must then be num_kv_heads * head_dim; total_k is ignored.
 *                Pool rows past a sequence's last key are never used: the kernel zeroes
 *                them in shared memory, so stale or NaN contents do not leak in.
 * cu_seqlens_q, cu_seqlens_k: [num_seqs + 1] int32, non-decreasing, starting at 0.
 * max_seqlen_q, max_seqlen_k: upper bounds of Lq and Lk over the batch.
 * block_table:   NULL, or [num_seqs, block_table_width] int32.
 * workspace:     pkv_prefill_workspace_bytes(...) bytes, 16-byte aligned, private to this
 *                call while it runs (two calls that may overlap need two workspaces).
 * out:           [Tq, num_q_heads, head_dim] bf16, contiguous.
 * Implemented: head_dim == 128, block_size a multiple of 256 when block_table is given,
 * num_q_heads / num_kv_heads in {1, 2, 4, 8}, token strides that are multiples of 8 elements, and
 * 16-byte aligned q, k, v.
 */
pkv_status pkv_varlen_prefill_attn(const void *q, int64_t q_tok_stride, int64_t total_q,
                                   const void *k, const void *v, int64_t kv_tok_stride,
                                   int64_t total_k,
                                   const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                   int32_t num_seqs, int32_t max_seqlen_q, int32_t max_seqlen_k,
                                   const int32_t *block_table, int32_t block_table_width,
                                   int32_t block_size, int64_t num_blocks, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_dim, float scale,
                                   int32_t causal, void *workspace, size_t workspace_bytes,
                                   void *out, void *stream);

/*
 * paged_decode_attn_noalloc -- the same computation as pkv_paged_decode_attn, for callers
 * that cannot allocate device memory. (The nano-vLLM pages have no counterpart: this entry
 * point exists for library users, not for the method.)
 *
 * Who needs it: code that has no way to get a workspace at call time -- e.g. a plug-in in a
 * serving engine that has already given nearly all of HBM to its KV pool and offers kernels
 * no allocator, or a call site where cudaMalloc is not allowed (it synchronises the device,
 * and it is forbidden while a stream is being captured).
 *
 * Arguments are those of pkv_paged_decode_attn without workspace / workspace_bytes; the
 * caller still owns q, the pools, the tables and out. The split-K partial results live in a
 * fixed array of PKV_DECODE_NOALLOC_SCRATCH_BYTES bytes that belongs to the library's device
 * image, so every device that uses it holds that memory until the process exits. The split
 * plan is the one pkv_paged_decode_attn would use (same num_splits rule), so for the same
 * inputs the two entry points compute the same result. A problem whose plan needs more than
 * the array (pkv_decode_workspace_bytes(...) > PKV_DECODE_NOALLOC_SCRATCH_BYTES) is rejected
 * with PKV_ERR_WORKSPACE before anything is enqueued; choosing fewer splits (num_splits > 0)
 * or the workspace entry point avoids that. The automatic plan of the Qwen3-shaped batch (256
 * sequences x 16 query heads, contexts up to 2048) takes one split and needs only the 16-byte
 * header; two splits need about 4.2 MB.
 *
 * The first call on each device looks up the array's device address (cudaGetSymbolAddress,
 * with that device current) and caches it; make that first call before any stream capture.
 * A lookup that fails returns PKV_ERR_CUDA, is not cached (the next call tries again) and
 * leaves no pending CUDA error behind.
 * All calls on a device share the array. Its work counter starts at zero, and every call
 * leaves it at zero again (as with a workspace). Calls whose kernels may run at the same time
 * on the GPU (different streams without ordering) race on the array: order them on one
 * stream.
 */
#define PKV_DECODE_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

pkv_status pkv_paged_decode_attn_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                         const int32_t *block_tables, int32_t block_table_width,
                                         const int32_t *context_lens, int32_t batch,
                                         int32_t max_context_len, int32_t num_q_heads,
                                         int32_t num_kv_heads, int32_t head_dim,
                                         int32_t block_size, int64_t num_blocks, float scale,
                                         int32_t num_splits, void *out, void *stream);

/*
 * qk_norm_rope_store -- the step before the store, fused into it: «nano-vLLM 最小化vLLM重新实现»,
 * 架构 6 模型 (the Qwen3 layer: RMSNorm of every query and key head -- QK 归一化 -- then RoPE;
 * 辅助层: RotaryEmbedding reads a precomputed cos/sin cache), and 架构 5 (K/V written into
 * the paged cache through slot_mapping).
 *
 * qkv:        [num_tokens, (Hq + 2 Hkv) * head_dim] bf16, token stride qkv_tok_stride
 *             elements (a multiple of 8): Hq query heads, then Hkv key heads, then Hkv value
 *             heads (the fused projection's output).
 * positions:  [num_tokens] int64, the tokens' positions in their sequences.
 * q_norm_weight, k_norm_weight: [head_dim] bf16.   eps: >= 0.
 * cos_sin_cache: [max_position, head_dim] fp32; row p = cos of the half-dim angles of
 *             position p, then their sines.
 * For each query / key head x (fp32 arithmetic):
 *     n = bf16_rne(x * rsqrt(mean(x^2) + eps) * w)
 *     y_i = n_i c_i - n_{i+h} s_i,  y_{i+h} = n_{i+h} c_i + n_i s_i   (h = head_dim / 2,
 *                                    c, s = row positions[t] of the cache; rotate-half RoPE)
 * q_out [num_tokens, Hq, head_dim] bf16 (contiguous) gets the query heads' y (RNE); the key
 * heads' y and the value heads (unchanged) go to k_cache / v_cache row slot_mapping[t] exactly
 * as pkv_kv_store writes them (negative slot: nothing stored, q still written; slot >=
 * num_slots: skipped and PKV_DEVERR_SLOT_RANGE). A position outside [0, max_position) skips the
 * token's query and key heads and sets PKV_DEVERR_POSITION_RANGE.
 * Implemented: head_dim == 128, 16-byte aligned pointers, projection rows of at most 227 KiB
 * (one token's row is staged in shared memory). Asynchronous on `stream`.
 */
pkv_status pkv_qk_norm_rope_store(const void *qkv, int64_t qkv_tok_stride, int64_t num_tokens,
                                  const int64_t *positions, const void *q_norm_weight,
                                  const void *k_norm_weight, float eps,
                                  const float *cos_sin_cache, int64_t max_position,
                                  const int64_t *slot_mapping, void *q_out, void *k_cache,
                                  void *v_cache, int64_t num_slots, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, void *stream);

/* ------------------------------------------------------------------ block manager (host)
 *
 * The owner of the pool's blocks on the host: «nano-vLLM 最小化vLLM重新实现», 架构 3 (块管理器)
 * -- fixed-size blocks with a reference count and a hash, allocate() that reuses cached
 * prefix blocks by hash and takes new blocks only for the rest, xxhash over token ids,
 * preemption that frees a sequence's blocks; the per-sequence block list is the page table of
 * «企业官网建设流程全解析 (Nano-vLLM 指南)» §2.2, the cached prefix of its §4.4. It produces
 * the block tables that the attention calls read (slot of token i = table[i / block_size] *
 * block_size + i % block_size). Host memory only, no CUDA; one handle must not be used by
 * two threads at once. Rules:
 *   - Only full blocks are hashed: XXH64 (seed 0) of the previous block's hash (8 bytes,
 *     little-endian; absent for a sequence's first block) followed by the block's token ids
 *     (int32, little-endian). A hit also needs equal token ids.
 *   - Once a block of a sequence misses, the rest of the sequence gets new blocks.
 *   - Free blocks are handed out first-in first-out, 0, 1, 2, ... at the start; a freed block
 *     stays a possible hit until it is handed out again.
 */
typedef struct pkv_block_manager pkv_block_manager;

/* A manager of num_blocks blocks of block_size tokens, all free. NULL on bad sizes or when
 * out of host memory. Free it with pkv_bm_destroy. */
pkv_block_manager *pkv_bm_create(int32_t num_blocks, int32_t block_size);
void pkv_bm_destroy(pkv_block_manager *bm);

/* Free blocks (-1 for a NULL handle); a block's reference count (-1 for a bad id); a block's
 * hash, with *is_hashed = 0 for a block that is not full and registered. */
int32_t pkv_bm_num_free(const pkv_block_manager *bm);
int32_t pkv_bm_ref_count(const pkv_block_manager *bm, int32_t block);
pkv_status pkv_bm_block_hash(const pkv_block_manager *bm, int32_t block, uint64_t *hash,
                             int32_t *is_hashed);

/* Blocks for a new (or preempted and resumed) sequence of num_tokens tokens: writes
 * ceil(num_tokens / block_size) block ids to block_table (table_capacity entries available)
 * and their count to *num_table_blocks, and the number of leading tokens whose K/V are
 * already cached (a multiple of block_size) to *num_cached_tokens; a prefill then only has
 * to compute the rest. PKV_ERR_NO_BLOCKS, with nothing changed, when fewer free blocks than
 * ceil(num_tokens / block_size) are left. */
pkv_status pkv_bm_allocate(pkv_block_manager *bm, const int32_t *token_ids, int32_t num_tokens,
                           int32_t *block_table, int32_t table_capacity,
                           int32_t *num_table_blocks, int32_t *num_cached_tokens);

/* Release a finished or preempted sequence: each block's reference count drops by one (last
 * block first); blocks that reach zero go to the back of the free list. PKV_ERR_INVALID_ARG,
 * with nothing changed, for an id out of range or a block released more often than held. */
pkv_status pkv_bm_deallocate(pkv_block_manager *bm, const int32_t *block_table,
                             int32_t num_table_blocks);

/* 1 if a sequence that now has seq_len tokens (its newest token included) can be given the
 * block that token may need, else 0. */
int32_t pkv_bm_can_append(const pkv_block_manager *bm, int32_t seq_len);

/* After a token was appended (the sequence has seq_len tokens, token_ids holds all of them):
 * takes a new block when the token starts one (appended to block_table, *num_table_blocks
 * grows by one), and hashes and registers the last block when the token fills it. */
pkv_status pkv_bm_may_append(pkv_block_manager *bm, const int32_t *token_ids, int32_t seq_len,
                             int32_t *block_table, int32_t table_capacity,
                             int32_t *num_table_blocks);

/* XXH64 of len bytes (the hash the block manager uses), exported for tests. */
uint64_t pkv_xxh64(const void *data, size_t len, uint64_t seed);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
