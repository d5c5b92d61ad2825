// kv_store.cu -- scatter each new token's K and V rows into the paged pool via slot_mapping.
//
// The store of «nano-vLLM 最小化vLLM重新实现», 架构 5 (store_kvcache: K/V written into the
// paged cache through slot_mapping). Rows that are whole 16-byte multiples go through shared
// memory with 1-D bulk copies (one thread per token: K and V rows in, then out to the slot's
// pool rows), which keeps many tokens in flight on the TMA engine with no registers held.
// Longer rows use 16-byte vectors, one warp per token; unaligned rows go 2 bytes at a time.
//
// HBM traffic per token: 2 rows read + 2 rows written + 8 bytes of slot (algorithmic minimum).
#include <algorithm>

#include "device_common.cuh"
#include "launch.h"

namespace pkv {
namespace {

constexpr int kWarpsPerCta = 8;

// Rows staged through shared memory with 1-D bulk copies: lane i of a CTA moves token
// blockIdx.x * tokens_per_cta + i (its K row and V row in, both out to the slot's pool rows),
// so a CTA keeps up to 8 tokens in flight and the copies run on the TMA engine.
constexpr int kBulkTokensPerCta = 8;
__global__ void __launch_bounds__(32)
    kv_store_bulk_kernel(const uint8_t *__restrict__ k, int64_t k_stride, const uint8_t *__restrict__ v,
                         int64_t v_stride, const int64_t *__restrict__ slot_mapping,
                         int64_t num_tokens, uint8_t *__restrict__ k_cache,
                         uint8_t *__restrict__ v_cache, int64_t num_slots, uint32_t row_bytes,
                         int tokens_per_cta, unsigned int *err) {
  extern __shared__ __align__(128) uint8_t buf[];  // tokens_per_cta x (K row, V row)
  __shared__ uint64_t full[kBulkTokensPerCta];
  const int i = threadIdx.x;
  const int64_t t = (int64_t)blockIdx.x * tokens_per_cta + i;
  if (i >= tokens_per_cta || t >= num_tokens) return;
  const int64_t slot = __ldg(slot_mapping + t);
  if (slot < 0) return;
  if (slot >= num_slots) {
    record_error(err, 1u /* PKV_DEVERR_SLOT_RANGE */);
    return;
  }
  if (aborted(err)) return;  // an earlier wait gave up somewhere: issue nothing
  uint8_t *kb = buf + (size_t)i * 2 * row_bytes, *vb = kb + row_bytes;
  mbar_init(&full[i], 1);  // this thread's own barrier: no other thread touches it
  fence_mbar_init();
  mbar_arrive_expect_tx(&full[i], 2 * row_bytes);
  bulk_copy_g2s(kb, k + t * k_stride, row_bytes, &full[i]);
  bulk_copy_g2s(vb, v + t * v_stride, row_bytes, &full[i]);
  // the rows are this thread's own copies: wait for them to land even if another CTA has
  // given up meanwhile (only the time limit ends this wait)
  if (!wait_own(&full[i], 0, err)) return;
  bulk_copy_s2g(k_cache + slot * row_bytes, kb, row_bytes);
  bulk_copy_s2g(v_cache + slot * row_bytes, vb, row_bytes);
  bulk_commit();
  bulk_wait_read_all();  // the rows must stay in shared memory until the copies have read them
}

// Any row length that is a whole number of 16-byte vectors.
__global__ void __launch_bounds__(kWarpsPerCta * 32)
    kv_store_vec_kernel(const uint4 *__restrict__ k, int64_t k_stride, const uint4 *__restrict__ v,
                        int64_t v_stride, const int64_t *__restrict__ slot_mapping,
                        int64_t num_tokens, uint4 *__restrict__ k_cache,
                        uint4 *__restrict__ v_cache, int64_t num_slots, int64_t row,
                        unsigned int *err) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerCta;
  for (int64_t t = warp0; t < num_tokens; t += nwarps) {
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (lane == 0) record_error(err, 1u);
      continue;
    }
    for (int64_t i = lane; i < row; i += 32) {
      k_cache[slot * row + i] = ld_stream_u4(k + t * k_stride + i);
      v_cache[slot * row + i] = ld_stream_u4(v + t * v_stride + i);
    }
  }
}

// Fallback for rows or addresses that are not 16-byte multiples: one bf16 at a time.
__global__ void __launch_bounds__(kWarpsPerCta * 32)
    kv_store_u16_kernel(const uint16_t *__restrict__ k, int64_t k_stride,
                        const uint16_t *__restrict__ v, int64_t v_stride,
                        const int64_t *__restrict__ slot_mapping, int64_t num_tokens,
                        uint16_t *__restrict__ k_cache, uint16_t *__restrict__ v_cache,
                        int64_t num_slots, int64_t row, unsigned int *err) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerCta;
  for (int64_t t = warp0; t < num_tokens; t += nwarps) {
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (lane == 0) record_error(err, 1u);
      continue;
    }
    for (int64_t i = lane; i < row; i += 32) {
      k_cache[slot * row + i] = k[t * k_stride + i];
      v_cache[slot * row + i] = v[t * v_stride + i];
    }
  }
}

}  // namespace

cudaError_t launch_kv_store(const void *k, int64_t k_tok_stride, const void *v,
                            int64_t v_tok_stride, const int64_t *slot_mapping, int64_t num_tokens,
                            void *k_cache, void *v_cache, int64_t num_slots, int64_t row_elems,
                            unsigned int *err, int num_sms, cudaStream_t stream) {
  const int64_t warps_needed = num_tokens;
  const int64_t max_ctas = (int64_t)num_sms * 8;  // 8 CTAs x 8 warps = 64 warps per SM
  const int64_t ctas64 = (warps_needed + kWarpsPerCta - 1) / kWarpsPerCta;
  const unsigned int ctas = (unsigned int)(ctas64 < max_ctas ? ctas64 : max_ctas);
  const dim3 block(kWarpsPerCta * 32);

  auto aligned16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const bool vec_ok = (row_elems % 8 == 0) && (k_tok_stride % 8 == 0) && (v_tok_stride % 8 == 0) &&
                      aligned16(k) && aligned16(v) && aligned16(k_cache) && aligned16(v_cache);
  const int64_t row_bytes = row_elems * 2;
  const int64_t bulk_tpc = row_bytes > 0 ? std::min<int64_t>(kBulkTokensPerCta, (96 * 1024) / (2 * row_bytes)) : 0;
  if (vec_ok && bulk_tpc >= 1) {
    const int64_t smem = bulk_tpc * 2 * row_bytes;
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (smem > 48 * 1024 && (dev >= 64 || !configured[dev])) {
      const cudaError_t e = cudaFuncSetAttribute(
          kv_store_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
      if (e != cudaSuccess) return e;
      if (dev < 64) configured[dev] = true;
    }
    const int64_t grid = (num_tokens + bulk_tpc - 1) / bulk_tpc;
    if (grid > INT32_MAX) return cudaErrorInvalidValue;
    kv_store_bulk_kernel<<<(unsigned)grid, 32, (size_t)smem, stream>>>(
        static_cast<const uint8_t *>(k), k_tok_stride * 2, static_cast<const uint8_t *>(v),
        v_tok_stride * 2, slot_mapping, num_tokens, static_cast<uint8_t *>(k_cache),
        static_cast<uint8_t *>(v_cache), num_slots, (uint32_t)row_bytes, (int)bulk_tpc, err);
  } else if (vec_ok) {  // rows too long to stage: 16-byte vectors straight through
    kv_store_vec_kernel<<<ctas, block, 0, stream>>>(
        static_cast<const uint4 *>(k), k_tok_stride / 8, static_cast<const uint4 *>(v),
        v_tok_stride / 8, slot_mapping, num_tokens, static_cast<uint4 *>(k_cache),
        static_cast<uint4 *>(v_cache), num_slots, row_elems / 8, err);
  } else {
    kv_store_u16_kernel<<<ctas, block, 0, stream>>>(
        static_cast<const uint16_t *>(k), k_tok_stride, static_cast<const uint16_t *>(v),
        v_tok_stride, slot_mapping, num_tokens, static_cast<uint16_t *>(k_cache),
        static_cast<uint16_t *>(v_cache), num_slots, row_elems, err);
  }
  return cudaGetLastError();
}

}  // namespace pkv
