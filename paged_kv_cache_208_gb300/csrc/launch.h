// launch.h -- host-side launchers behind the C ABI (internal to libpkv).
//
// The extern "C" entry points in pkv_api.cu validate arguments and then call these; each
// launcher only enqueues kernels on `stream` and returns the launch status.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

// kv_store.cu
cudaError_t launch_kv_store(const void *k, int64_t k_tok_stride, const void *v,
                            int64_t v_tok_stride, const int64_t *slot_mapping, int64_t num_tokens,
                            void *k_cache, void *v_cache, int64_t num_slots, int64_t row_elems,
                            unsigned int *err, int num_sms, cudaStream_t stream);

// decode.cu
struct DecodePlan {
  int32_t chunk;       // logical tokens per split (multiple of 64)
  int32_t splits;      // splits of the longest context
  int32_t head_groups; // CTAs per KV head (query heads handled two at a time)
  int32_t heads_per_cta;
  size_t workspace_bytes;
};
DecodePlan plan_decode(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t max_context_len, int32_t num_splits, int num_sms);

struct DecodeArgs {
  const void *q;
  const void *k_cache;
  const void *v_cache;
  const int32_t *block_tables;
  int32_t table_width;
  const int32_t *context_lens;
  int32_t batch;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t block_size;
  int64_t num_blocks;
  float scale;
  void *workspace;
  void *out;
  unsigned int *err;
  int num_sms;
  // optional: the step's new tokens, stored into the pools before they are read (one per
  // sequence, [batch, num_kv_heads, 128] with these token strides, at slot_mapping[b])
  const void *k_new = nullptr;
  const void *v_new = nullptr;
  int64_t k_new_stride = 0;
  int64_t v_new_stride = 0;
  const int64_t *slot_mapping = nullptr;
  int64_t num_slots = 0;
};
constexpr size_t kDecodeQueueBytes = 16;  // the workspace's header: the work counters
cudaError_t launch_paged_decode(const DecodeArgs &a, const DecodePlan &plan,
                                cudaStream_t stream);

// prefill.cu
struct PrefillArgs {
  const void *q;
  int64_t q_tok_stride;
  int64_t total_q;   // rows of q (and of out)
  const void *k;
  const void *v;
  int64_t kv_tok_stride;
  int64_t kv_rows;   // rows addressable through k/v (Tk, or num_blocks * block_size)
  const int32_t *cu_seqlens_q;
  const int32_t *cu_seqlens_k;
  int32_t num_seqs;
  int32_t max_seqlen_q;
  int32_t max_seqlen_k;
  const int32_t *block_table;
  int32_t table_width;
  int32_t block_size;
  int64_t num_blocks;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  float scale;
  int32_t causal;
  void *out;
  void *workspace;   // prefill_workspace_layout(...).bytes: the work list and its counter
  unsigned int *err;
};

// The prefill workspace: a 16-byte header (work counter, number of work units), the
// per-sequence query-block counts, the sequences ranked by that count, the first unit of each
// ranked sequence, two histograms over the counts, and the unit list itself -- one
// (sequence, query block) pair per unit, at most num_seqs * ceil(max_seqlen_q / 128).
struct PrefillWorkspace {
  size_t counts, ranked, unit_start, hist, fill, units, bytes;
  int64_t max_units;
  int32_t levels;  // ceil(max_seqlen_q / 128): the query blocks of the longest sequence
};
inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }
inline PrefillWorkspace prefill_workspace_layout(int32_t num_seqs, int32_t max_seqlen_q) {
  PrefillWorkspace w{};
  w.levels = (int32_t)(((int64_t)max_seqlen_q + 127) / 128);
  w.max_units = (int64_t)num_seqs * w.levels;
  const size_t n = (size_t)num_seqs, l = (size_t)w.levels + 1;
  w.counts = 16;
  w.ranked = align16(w.counts + 4 * n);
  w.unit_start = align16(w.ranked + 4 * n);
  w.hist = align16(w.unit_start + 4 * (n + 1));
  w.fill = align16(w.hist + 4 * l);
  w.units = align16(w.fill + 4 * l);
  w.bytes = align16(w.units + 8 * (size_t)w.max_units);
  return w;
}
cudaError_t launch_varlen_prefill(const PrefillArgs &a, int num_sms, cudaStream_t stream);
bool prefill_group_supported(int group);  // num_q_heads / num_kv_heads

// the current device's SM count and the address of the device error word (pkv_api.cu);
// 0 / nullptr when the CUDA runtime cannot answer
int current_sm_count();
unsigned int *current_error_word();

// tensor maps (pkv_api.cu): the driver's cuTensorMapEncodeTiled, fetched at run time
CUresult encode_tensor_map(CUtensorMap *map, CUtensorMapDataType dtype, uint32_t rank,
                           void *base, const uint64_t *dims, const uint64_t *strides_bytes,
                           const uint32_t *box, CUtensorMapSwizzle swizzle,
                           CUtensorMapL2promotion promotion);

}  // namespace pkv
