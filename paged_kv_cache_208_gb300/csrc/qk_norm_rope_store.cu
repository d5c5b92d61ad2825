// qk_norm_rope_store.cu -- the step just before the store, fused into it: RMSNorm of every
// query and key head, rotary position embedding, and the store of K and V into the paged pool.
//
// «nano-vLLM 最小化vLLM重新实现», 架构 6 模型: the Qwen3 layer normalises every query and key
// head with an RMSNorm (QK 归一化) and applies RoPE; 辅助层: RotaryEmbedding reads a
// precomputed cos/sin cache; 架构 5: the K/V that come out are written into the paged cache
// through slot_mapping. Doing all of it in one pass reads the projection output once and
// writes q and the cache rows once (instead of norm, RoPE and store each reading and writing
// K again).
//
// Token t's projection row holds Hq query heads, Hkv key heads and Hkv value heads of 128
// values. For a query or key head x with weight w, in fp32:
//     n = bf16(x * rsqrt(mean(x^2) + eps) * w)          (the normalised activation, bf16)
//     y_i = n_i c_i - n_{i+64} s_i,  y_{i+64} = n_{i+64} c_i + n_i s_i,  i < 64
// with c = cos_sin[pos, 0:64], s = cos_sin[pos, 64:128], rounded to bf16 (RNE): query heads
// to q_out, key heads to k_cache[slot]; value heads are copied to v_cache[slot] bit for bit.
//
// A quarter warp (8 lanes) owns one head row: lane l holds elements 8l..8l+7 and their RoPE
// partners 64+8l..64+8l+7 (16-byte loads and stores), so the rotation needs no exchange and
// the sum of squares takes three shuffles. A warp does four rows; HBM traffic per token is
// its projection row in and q, K and V out.
#include <math.h>
#include <stdint.h>

#include "device_common.cuh"
#include "launch.h"
#include "pkv.h"

namespace pkv {
namespace {

constexpr int kD = 128;
constexpr int kHalf = kD / 2;
constexpr int kThreads = 256;
constexpr int kRowsPerWarp = 4;

struct RopeParams {
  const uint16_t *qkv;
  int64_t tok_stride;  // elements
  int64_t num_tokens;
  const int64_t *positions;
  const uint16_t *q_weight;
  const uint16_t *k_weight;
  float eps;
  const float *cos_sin;
  int64_t max_position;
  const int64_t *slots;
  uint16_t *q_out;
  uint16_t *k_cache;
  uint16_t *v_cache;
  int64_t num_slots;
  int32_t hq, hkv;
  unsigned int *err;
};

__device__ __forceinline__ float bf(uint32_t bits16) { return __uint_as_float(bits16 << 16); }
__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf(w[i] & 0xFFFFu);
    f[2 * i + 1] = bf(w[i] >> 16);
  }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = (uint32_t)bf16_bits_rn(f[2 * i]) | ((uint32_t)bf16_bits_rn(f[2 * i + 1]) << 16);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__global__ void __launch_bounds__(kThreads) qk_norm_rope_store_kernel(const RopeParams p) {
  const int lane = threadIdx.x & 31;
  const int group = lane >> 3, gl = lane & 7;
  const int heads = p.hq + 2 * p.hkv;
  const int64_t row = ((int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5)) *
                          kRowsPerWarp + group;
  const bool live = row < p.num_tokens * heads;
  const int64_t t = live ? row / heads : 0;
  const int h = live ? (int)(row % heads) : 0;
  const uint16_t *src = p.qkv + t * p.tok_stride + (int64_t)h * kD;
  const uint4 *lo_src = reinterpret_cast<const uint4 *>(src + 8 * gl);
  const uint4 *hi_src = reinterpret_cast<const uint4 *>(src + kHalf + 8 * gl);
  const int64_t slot = live && h >= p.hq ? p.slots[t] : -1;
  const bool slot_ok = slot >= 0 && slot < p.num_slots;
  if (live && h >= p.hq && slot >= p.num_slots && gl == 0) record_error(p.err, 1u /* SLOT */);

  // every lane loads and joins the shuffles before any lane leaves (full-warp shuffles)
  const uint4 lo = live ? ld_stream_u4(lo_src) : make_uint4(0, 0, 0, 0);
  const uint4 hi = live ? ld_stream_u4(hi_src) : make_uint4(0, 0, 0, 0);
  float a[8], b[8];
  unpack8(lo, a);
  unpack8(hi, b);
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) ss = fmaf(a[i], a[i], fmaf(b[i], b[i], ss));
  // the quarter warp's sum (lanes 8g..8g+7)
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  ss += __shfl_xor_sync(0xffffffffu, ss, 2);
  ss += __shfl_xor_sync(0xffffffffu, ss, 4);
  if (!live) return;
  if (h >= p.hq + p.hkv) {  // value head: straight copy
    if (slot_ok) {
      uint16_t *dst = p.v_cache + slot * ((int64_t)p.hkv * kD) + (int64_t)(h - p.hq - p.hkv) * kD;
      reinterpret_cast<uint4 *>(dst + 8 * gl)[0] = lo;
      reinterpret_cast<uint4 *>(dst + kHalf + 8 * gl)[0] = hi;
    }
    return;
  }
  const int64_t pos = p.positions[t];
  if (pos < 0 || pos >= p.max_position) {
    if (gl == 0) record_error(p.err, 32u /* POSITION_RANGE */);
    return;
  }
  const bool is_q = h < p.hq;
  if (!is_q && !slot_ok) return;
  const float r = rsqrtf(ss * (1.f / kD) + p.eps);
  const uint16_t *wsrc = is_q ? p.q_weight : p.k_weight;
  float wa[8], wb[8];
  unpack8(*reinterpret_cast<const uint4 *>(wsrc + 8 * gl), wa);
  unpack8(*reinterpret_cast<const uint4 *>(wsrc + kHalf + 8 * gl), wb);
  const float4 *cs = reinterpret_cast<const float4 *>(p.cos_sin + pos * kD);
  const float4 c0 = cs[2 * gl], c1 = cs[2 * gl + 1];
  const float4 s0 = cs[16 + 2 * gl], s1 = cs[16 + 2 * gl + 1];
  const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  float ya[8], yb[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    // the normalised activation is bf16, as between the model's layers
    const float na = bf(bf16_bits_rn(a[i] * r * wa[i]));
    const float nb = bf(bf16_bits_rn(b[i] * r * wb[i]));
    ya[i] = na * c[i] - nb * s[i];
    yb[i] = nb * c[i] + na * s[i];
  }
  uint16_t *dst = is_q ? p.q_out + (t * p.hq + h) * kD
                       : p.k_cache + slot * ((int64_t)p.hkv * kD) + (int64_t)(h - p.hq) * kD;
  reinterpret_cast<uint4 *>(dst + 8 * gl)[0] = pack8(ya);
  reinterpret_cast<uint4 *>(dst + kHalf + 8 * gl)[0] = pack8(yb);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_qk_norm_rope_store(
    const void *qkv, int64_t qkv_tok_stride, int64_t num_tokens, const int64_t *positions,
    const void *q_norm_weight, const void *k_norm_weight, float eps,
    const float *cos_sin_cache, int64_t max_position, const int64_t *slot_mapping, void *q_out,
    void *k_cache, void *v_cache, int64_t num_slots, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, void *stream) {
  using namespace pkv;
  if (num_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      num_slots < 0 || max_position <= 0 || !(eps >= 0.f) || !isfinite(eps))
    return PKV_ERR_INVALID_ARG;
  if (qkv_tok_stride < (int64_t)(num_q_heads + 2 * num_kv_heads) * head_dim)
    return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!qkv || !positions || !q_norm_weight || !k_norm_weight || !cos_sin_cache ||
      !slot_mapping || !q_out || !k_cache || !v_cache)
    return PKV_ERR_INVALID_ARG;
  if (head_dim != kD) return PKV_ERR_UNSUPPORTED;
  if (qkv_tok_stride % 8 != 0 || !aligned16(qkv) || !aligned16(q_norm_weight) ||
      !aligned16(k_norm_weight) || !aligned16(cos_sin_cache) || !aligned16(q_out) ||
      !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_UNSUPPORTED;
  unsigned int *err = current_error_word();
  if (!err) return PKV_ERR_CUDA;
  const int64_t rows = num_tokens * (num_q_heads + 2 * num_kv_heads);
  const int64_t rows_per_cta = (kThreads / 32) * kRowsPerWarp;
  const int64_t grid = (rows + rows_per_cta - 1) / rows_per_cta;
  if (grid > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  RopeParams prm{};
  prm.qkv = static_cast<const uint16_t *>(qkv);
  prm.tok_stride = qkv_tok_stride;
  prm.num_tokens = num_tokens;
  prm.positions = positions;
  prm.q_weight = static_cast<const uint16_t *>(q_norm_weight);
  prm.k_weight = static_cast<const uint16_t *>(k_norm_weight);
  prm.eps = eps;
  prm.cos_sin = cos_sin_cache;
  prm.max_position = max_position;
  prm.slots = slot_mapping;
  prm.q_out = static_cast<uint16_t *>(q_out);
  prm.k_cache = static_cast<uint16_t *>(k_cache);
  prm.v_cache = static_cast<uint16_t *>(v_cache);
  prm.num_slots = num_slots;
  prm.hq = num_q_heads;
  prm.hkv = num_kv_heads;
  prm.err = err;
  qk_norm_rope_store_kernel<<<(unsigned)grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      prm);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
