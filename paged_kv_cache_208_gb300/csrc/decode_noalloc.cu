// decode_noalloc.cu -- paged decode attention for callers that cannot allocate device memory.
//
// pkv_paged_decode_attn needs a caller-provided workspace for the split-K partial results.
// Some callers cannot provide one: a plug-in inside a serving engine that has already handed
// nearly all of HBM to its KV pool and exposes no allocator to kernels, or code that may not
// call cudaMalloc at that point (it synchronises the device, and is not allowed while a
// stream is being captured). This entry point takes the same inputs and outputs and keeps
// the partial results in a fixed-size array that is part of this library's device image.
//
// The array is shared by every call on a device and keeps whatever the last call left in it;
// the kernels write every partial they later read, so nothing has to start at zero. Two
// calls whose kernels overlap on the GPU (different streams, no ordering between them) race
// on the array and give wrong results: order them on one stream, or use the workspace entry
// point.
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "launch.h"
#include "pkv.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PKV_DECODE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

struct ScratchSlot {
  std::mutex mu;
  void *ptr = nullptr;
};
ScratchSlot g_scratch[kMaxDevices];

// The device address of the scratch array on the current device. In host code the array's
// name is only a host-side stand-in, so the address is looked up (with that device current)
// and cached. Only a successful lookup is cached: a failed one (for example made while a
// stream is being captured) is retried by the next call, and its error is cleared so that
// it does not surface in the caller's next cudaGetLastError.
void *scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  ScratchSlot &s = g_scratch[dev];
  std::lock_guard<std::mutex> lock(s.mu);
  if (!s.ptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) == cudaSuccess && p != nullptr) {
      s.ptr = p;
    } else {
      (void)cudaGetLastError();
    }
  }
  return s.ptr;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" pkv_status pkv_paged_decode_attn_noalloc(
    const void *q, const void *k_cache, const void *v_cache, const int32_t *block_tables,
    int32_t block_table_width, const int32_t *context_lens, int32_t batch,
    int32_t max_context_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, int64_t num_blocks, float scale, int32_t num_splits, void *out,
    void *stream) {
  if (batch < 0 || max_context_len < 0 || num_splits < 0 || num_q_heads <= 0 ||
      num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 ||
      block_size <= 0 || num_blocks <= 0 || block_table_width <= 0 || !isfinite(scale))
    return PKV_ERR_INVALID_ARG;
  if (batch == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return PKV_ERR_INVALID_ARG;
  if (head_dim != 128 || block_size % 256 != 0) return PKV_ERR_UNSUPPORTED;
  if (num_blocks * (int64_t)block_size > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PKV_ERR_UNSUPPORTED;
  const int num_sms = pkv::current_sm_count();
  unsigned int *err = pkv::current_error_word();
  if (num_sms <= 0 || !err) return PKV_ERR_CUDA;
  const pkv::DecodePlan plan =
      pkv::plan_decode(batch, num_q_heads, num_kv_heads, max_context_len, num_splits, num_sms);
  if (plan.workspace_bytes > PKV_DECODE_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
  void *scratch = scratch_on_current_device();  // the first call on a device looks it up
  if (!scratch) return PKV_ERR_CUDA;
  pkv::DecodeArgs a{q,           k_cache,      v_cache,     block_tables, block_table_width,
                    context_lens, batch,        num_q_heads, num_kv_heads, block_size,
                    num_blocks,  scale,        scratch,     out,          err,
                    num_sms};
  return pkv::launch_paged_decode(a, plan, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}
