// pkv_api.cu -- the extern "C" entry points of libpkv: argument checks, split planning,
// tensor-map encoding and the device-side error word. No entry point allocates memory or
// synchronises the host, except the pkv_get_device_errors diagnostic.
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "launch.h"
#include "pkv.h"

namespace {

__device__ unsigned int g_device_errors;

constexpr int kMaxDevices = 64;

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

// Per-device facts looked up once: SM count and the address of the error word.
struct DeviceInfo {
  std::once_flag once;
  int num_sms = 0;
  unsigned int *err = nullptr;
  bool ok = false;
};
DeviceInfo g_devices[kMaxDevices];

DeviceInfo *device_info() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceInfo &d = g_devices[dev];
  std::call_once(d.once, [&] {
    void *p = nullptr;
    d.ok = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
           cudaGetSymbolAddress(&p, g_device_errors) == cudaSuccess;
    d.err = static_cast<unsigned int *>(p);
  });
  return d.ok ? &d : nullptr;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

pkv_status launch_status(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

}  // namespace

namespace pkv {

int current_sm_count() {
  DeviceInfo *d = device_info();
  return d ? d->num_sms : 0;
}

unsigned int *current_error_word() {
  DeviceInfo *d = device_info();
  return d ? d->err : nullptr;
}

CUresult encode_tensor_map(CUtensorMap *map, CUtensorMapDataType dtype, uint32_t rank,
                           void *base, const uint64_t *dims, const uint64_t *strides_bytes,
                           const uint32_t *box, CUtensorMapSwizzle swizzle,
                           CUtensorMapL2promotion promotion) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return CUDA_ERROR_NOT_SUPPORTED;
  cuuint64_t gdim[5], gstride[4];
  cuuint32_t bdim[5], estride[5];
  for (uint32_t i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
    if (i + 1 < rank) gstride[i] = strides_bytes[i];
  }
  return fn(map, dtype, rank, base, gdim, gstride, bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle, promotion, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace pkv

extern "C" {

const char *pkv_status_string(pkv_status status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape or layout";
    case PKV_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case PKV_ERR_CUDA: return "CUDA call failed";
    case PKV_ERR_NO_BLOCKS: return "not enough free blocks";
    default: return "unknown status";
  }
}

int32_t pkv_abi_version(void) { return 2; }

pkv_status pkv_raise_device_errors(uint32_t bits) {
  if (!device_info()) return PKV_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return PKV_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_errors, sizeof v) != cudaSuccess) return PKV_ERR_CUDA;
  v |= bits;
  if (cudaMemcpyToSymbol(g_device_errors, &v, sizeof v) != cudaSuccess) return PKV_ERR_CUDA;
  return PKV_OK;
}

pkv_status pkv_get_device_errors(uint32_t *errors, int32_t reset) {
  if (!errors) return PKV_ERR_INVALID_ARG;
  if (!device_info()) return PKV_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return PKV_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_errors, sizeof v) != cudaSuccess) return PKV_ERR_CUDA;
  *errors = v;
  if (reset) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_device_errors, &zero, sizeof zero) != cudaSuccess)
      return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

pkv_status pkv_kv_store(const void *k, int64_t k_tok_stride, const void *v, int64_t v_tok_stride,
                        const int64_t *slot_mapping, int64_t num_tokens, void *k_cache,
                        void *v_cache, int64_t num_slots, int32_t num_kv_heads,
                        int32_t head_dim, void *stream) {
  if (num_tokens < 0 || num_slots < 0 || num_kv_heads <= 0 || head_dim <= 0)
    return PKV_ERR_INVALID_ARG;
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  if (k_tok_stride < row || v_tok_stride < row) return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
  DeviceInfo *dev = device_info();
  if (!dev) return PKV_ERR_CUDA;
  return launch_status(pkv::launch_kv_store(k, k_tok_stride, v, v_tok_stride, slot_mapping,
                                            num_tokens, k_cache, v_cache, num_slots, row, dev->err,
                                            dev->num_sms, static_cast<cudaStream_t>(stream)));
}

size_t pkv_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_context_len,
                                  int32_t num_splits) {
  if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 ||
      head_dim != 128 || max_context_len < 0 || num_splits < 0)
    return 0;
  DeviceInfo *dev = device_info();
  if (!dev) return 0;
  return pkv::plan_decode(batch, num_q_heads, num_kv_heads, max_context_len, num_splits,
                          dev->num_sms)
      .workspace_bytes;
}

pkv_status pkv_paged_decode_attn(const void *q, const void *k_cache, const void *v_cache,
                                 const int32_t *block_tables, int32_t block_table_width,
                                 const int32_t *context_lens, int32_t batch,
                                 int32_t max_context_len, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                 int64_t num_blocks, float scale, int32_t num_splits,
                                 void *workspace, size_t workspace_bytes, void *out,
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
  DeviceInfo *dev = device_info();
  if (!dev) return PKV_ERR_CUDA;
  const pkv::DecodePlan plan = pkv::plan_decode(batch, num_q_heads, num_kv_heads,
                                                max_context_len, num_splits, dev->num_sms);
  if (!workspace || workspace_bytes < plan.workspace_bytes || !aligned16(workspace))
    return PKV_ERR_WORKSPACE;
  pkv::DecodeArgs a{q,           k_cache,        v_cache,      block_tables, block_table_width,
                    context_lens, batch,          num_q_heads,  num_kv_heads, block_size,
                    num_blocks,  scale,          workspace,    out,          dev->err,
                    dev->num_sms};
  return launch_status(pkv::launch_paged_decode(a, plan, static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_paged_decode_step(const void *q, const void *k_new, int64_t k_new_tok_stride,
                                 const void *v_new, int64_t v_new_tok_stride,
                                 const int64_t *slot_mapping, void *k_cache, void *v_cache,
                                 const int32_t *block_tables, int32_t block_table_width,
                                 const int32_t *context_lens, int32_t batch,
                                 int32_t max_context_len, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                 int64_t num_blocks, float scale, int32_t num_splits,
                                 void *workspace, size_t workspace_bytes, void *out,
                                 void *stream) {
  if (batch < 0 || max_context_len < 0 || num_splits < 0 || num_q_heads <= 0 ||
      num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 ||
      block_size <= 0 || num_blocks <= 0 || block_table_width <= 0 || !isfinite(scale))
    return PKV_ERR_INVALID_ARG;
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  if (k_new_tok_stride < row || v_new_tok_stride < row) return PKV_ERR_INVALID_ARG;
  if (batch == 0) return PKV_OK;
  if (!q || !k_new || !v_new || !slot_mapping || !k_cache || !v_cache || !block_tables ||
      !context_lens || !out)
    return PKV_ERR_INVALID_ARG;
  if (head_dim != 128 || block_size % 256 != 0) return PKV_ERR_UNSUPPORTED;
  if (num_blocks * (int64_t)block_size > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      !aligned16(k_new) || !aligned16(v_new) || k_new_tok_stride % 8 != 0 ||
      v_new_tok_stride % 8 != 0)
    return PKV_ERR_UNSUPPORTED;
  DeviceInfo *dev = device_info();
  if (!dev) return PKV_ERR_CUDA;
  const pkv::DecodePlan plan = pkv::plan_decode(batch, num_q_heads, num_kv_heads,
                                                max_context_len, num_splits, dev->num_sms);
  if (!workspace || workspace_bytes < plan.workspace_bytes || !aligned16(workspace))
    return PKV_ERR_WORKSPACE;
  pkv::DecodeArgs a{q,           k_cache,        v_cache,      block_tables, block_table_width,
                    context_lens, batch,          num_q_heads,  num_kv_heads, block_size,
                    num_blocks,  scale,          workspace,    out,          dev->err,
                    dev->num_sms};
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_new_stride = k_new_tok_stride;
  a.v_new_stride = v_new_tok_stride;
  a.slot_mapping = slot_mapping;
  a.num_slots = num_blocks * block_size;
  return launch_status(pkv::launch_paged_decode(a, plan, static_cast<cudaStream_t>(stream)));
}

size_t pkv_prefill_workspace_bytes(int32_t num_seqs, int32_t max_seqlen_q, int32_t num_q_heads,
                                   int32_t head_dim) {
  if (num_seqs < 0 || max_seqlen_q < 0 || num_q_heads <= 0 || head_dim <= 0) return 0;
  const pkv::PrefillWorkspace w = pkv::prefill_workspace_layout(num_seqs, max_seqlen_q);
  if (w.max_units > INT32_MAX) return 0;
  return w.bytes;
}

pkv_status pkv_varlen_prefill_attn(const void *q, int64_t q_tok_stride, int64_t total_q,
                                   const void *k, const void *v, int64_t kv_tok_stride,
                                   int64_t total_k,
                                   const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                   int32_t num_seqs, int32_t max_seqlen_q, int32_t max_seqlen_k,
                                   const int32_t *block_table, int32_t block_table_width,
                                   int32_t block_size, int64_t num_blocks, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_dim, float scale,
                                   int32_t causal, void *workspace, size_t workspace_bytes,
                                   void *out, void *stream) {
  if (num_seqs < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || num_q_heads <= 0 ||
      num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 ||
      !isfinite(scale))
    return PKV_ERR_INVALID_ARG;
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  if (q_tok_stride < (int64_t)num_q_heads * head_dim || kv_tok_stride < row)
    return PKV_ERR_INVALID_ARG;
  if (block_table && (block_size <= 0 || num_blocks <= 0 || block_table_width <= 0))
    return PKV_ERR_INVALID_ARG;
  if (total_q < 0 || (!block_table && total_k < 0)) return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0 || max_seqlen_q == 0 || total_q == 0) return PKV_OK;
  if (!q || !k || !v || !cu_seqlens_q || !cu_seqlens_k || !out) return PKV_ERR_INVALID_ARG;
  if (head_dim != 128 || !pkv::prefill_group_supported(num_q_heads / num_kv_heads))
    return PKV_ERR_UNSUPPORTED;
  if (block_table && (block_size % 256 != 0 || kv_tok_stride != row ||
                      num_blocks * (int64_t)block_size > INT32_MAX))
    return PKV_ERR_UNSUPPORTED;
  if (total_q > INT32_MAX || (!block_table && total_k > INT32_MAX)) return PKV_ERR_UNSUPPORTED;
  if (q_tok_stride % 8 != 0 || kv_tok_stride % 8 != 0 || !aligned16(q) || !aligned16(k) ||
      !aligned16(v) || !aligned16(out))
    return PKV_ERR_UNSUPPORTED;
  const pkv::PrefillWorkspace wl = pkv::prefill_workspace_layout(num_seqs, max_seqlen_q);
  if (wl.max_units > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < wl.bytes || !aligned16(workspace))
    return PKV_ERR_WORKSPACE;
  DeviceInfo *dev = device_info();
  if (!dev) return PKV_ERR_CUDA;
  pkv::PrefillArgs a{};
  a.q = q;
  a.q_tok_stride = q_tok_stride;
  a.total_q = total_q;
  a.kv_rows = block_table ? num_blocks * block_size : total_k;
  a.k = k;
  a.v = v;
  a.kv_tok_stride = kv_tok_stride;
  a.cu_seqlens_q = cu_seqlens_q;
  a.cu_seqlens_k = cu_seqlens_k;
  a.num_seqs = num_seqs;
  a.max_seqlen_q = max_seqlen_q;
  a.max_seqlen_k = max_seqlen_k;
  a.block_table = block_table;
  a.table_width = block_table_width;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.scale = scale;
  a.causal = causal;
  a.out = out;
  a.workspace = workspace;
  a.err = dev->err;
  return launch_status(pkv::launch_varlen_prefill(a, dev->num_sms,
                                                  static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
