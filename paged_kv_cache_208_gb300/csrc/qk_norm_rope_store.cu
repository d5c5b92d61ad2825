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
// A quarter warp (8 lanes) owns a head row: lane l holds elements 8l..8l+7 and their RoPE
// partners 64+8l..64+8l+7 (16-byte loads and stores), so the rotation needs no exchange and
// the sum of squares takes three shuffles. A warp does eight consecutive heads of one token,
// two per quarter; HBM traffic per token is its projection row in and q, K and V out.
// Roundings to bf16 go two values per conversion instruction.
#include <math.h>
#include <stdint.h>

#include <cuda_bf16.h>

#include "device_common.cuh"
#include "launch.h"
#include "pkv.h"

namespace pkv {
namespace {

constexpr int kD = 128;
constexpr int kHalf = kD / 2;
constexpr int kThreads = 256;
constexpr int kRowsPerWarp = 4;     // quarter warps
constexpr int kRowsPerQuarter = 2;  // head rows each quarter warp processes

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
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
// two floats to a bf16 pair (RNE), one conversion instruction
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
}
// round to bf16 and back (the normalised activation is bf16, as between the model's layers)
__device__ __forceinline__ void round8(float (&f)[8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w = pack2(f[2 * i], f[2 * i + 1]);
    f[2 * i] = bf(w & 0xFFFFu);
    f[2 * i + 1] = __uint_as_float(w & 0xFFFF0000u);
  }
}

struct Row {
  bool live;
  int64_t t;
  int h;
  uint4 lo, hi;
  float ss;
};

__device__ __forceinline__ Row load_row(const RopeParams &p, int64_t t, int h, int heads,
                                        int gl) {
  Row r;
  r.live = t < p.num_tokens && h < heads;
  r.t = r.live ? t : 0;
  r.h = r.live ? h : 0;
  const uint16_t *src = p.qkv + r.t * p.tok_stride + (int64_t)r.h * kD;
  r.lo = r.live ? ld_stream_u4(reinterpret_cast<const uint4 *>(src + 8 * gl))
                : make_uint4(0, 0, 0, 0);
  r.hi = r.live ? ld_stream_u4(reinterpret_cast<const uint4 *>(src + kHalf + 8 * gl))
                : make_uint4(0, 0, 0, 0);
  return r;
}

// One head row after its sum of squares is known (no shuffles from here on).
__device__ __forceinline__ void finish_row(const RopeParams &p, const Row &r, int gl) {
  if (!r.live) return;
  const bool is_v = r.h >= p.hq + p.hkv, is_q = r.h < p.hq;
  const int64_t slot = is_q ? -1 : p.slots[r.t];
  const bool slot_ok = slot >= 0 && slot < p.num_slots;
  if (!is_q && slot >= p.num_slots && gl == 0) record_error(p.err, 1u /* SLOT_RANGE */);
  if (is_v) {  // value head: straight copy
    if (slot_ok) {
      uint16_t *dst =
          p.v_cache + slot * ((int64_t)p.hkv * kD) + (int64_t)(r.h - p.hq - p.hkv) * kD;
      reinterpret_cast<uint4 *>(dst + 8 * gl)[0] = r.lo;
      reinterpret_cast<uint4 *>(dst + kHalf + 8 * gl)[0] = r.hi;
    }
    return;
  }
  const int64_t pos = p.positions[r.t];
  if (pos < 0 || pos >= p.max_position) {
    if (gl == 0) record_error(p.err, 32u /* POSITION_RANGE */);
    return;
  }
  if (!is_q && !slot_ok) return;
  const float rs = rsqrtf(r.ss * (1.f / kD) + p.eps);
  const uint16_t *wsrc = is_q ? p.q_weight : p.k_weight;
  float a[8], b[8], wa[8], wb[8];
  unpack8(r.lo, a);
  unpack8(r.hi, b);
  unpack8(*reinterpret_cast<const uint4 *>(wsrc + 8 * gl), wa);
  unpack8(*reinterpret_cast<const uint4 *>(wsrc + kHalf + 8 * gl), wb);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    a[i] = a[i] * rs * wa[i];
    b[i] = b[i] * rs * wb[i];
  }
  round8(a);
  round8(b);
  const float4 *cs = reinterpret_cast<const float4 *>(p.cos_sin + pos * kD);
  const float4 c0 = cs[2 * gl], c1 = cs[2 * gl + 1];
  const float4 s0 = cs[16 + 2 * gl], s1 = cs[16 + 2 * gl + 1];
  const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  float ya[8], yb[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    ya[i] = a[i] * c[i] - b[i] * s[i];
    yb[i] = b[i] * c[i] + a[i] * s[i];
  }
  uint16_t *dst = is_q ? p.q_out + (r.t * p.hq + r.h) * kD
                       : p.k_cache + slot * ((int64_t)p.hkv * kD) + (int64_t)(r.h - p.hq) * kD;
  reinterpret_cast<uint4 *>(dst + 8 * gl)[0] = pack8(ya);
  reinterpret_cast<uint4 *>(dst + kHalf + 8 * gl)[0] = pack8(yb);
}

__device__ __forceinline__ float sum_sq(const uint4 lo, const uint4 hi) {
  float a[8], b[8];
  unpack8(lo, a);
  unpack8(hi, b);
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) ss = fmaf(a[i], a[i], fmaf(b[i], b[i], ss));
  return ss;
}

// A warp owns eight consecutive heads of one token; quarter warp g takes heads 8k + g and
// 8k + 4 + g. All four 16-byte loads are issued before any arithmetic, so each lane keeps 64
// bytes in flight. The token and head block come from one 32-bit division per warp.
__global__ void __launch_bounds__(kThreads, 4) qk_norm_rope_store_kernel(const RopeParams p,
                                                                       uint32_t warps_per_token) {
  const int lane = threadIdx.x & 31;
  const int group = lane >> 3, gl = lane & 7;
  const int heads = p.hq + 2 * p.hkv;
  const uint32_t wg = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  const uint32_t t = wg / warps_per_token;
  const int h0 = (int)(wg - t * warps_per_token) * (kRowsPerQuarter * kRowsPerWarp) + group;
  Row r0 = load_row(p, t, h0, heads, gl);
  Row r1 = load_row(p, t, h0 + kRowsPerWarp, heads, gl);
  r0.ss = sum_sq(r0.lo, r0.hi);
  r1.ss = sum_sq(r1.lo, r1.hi);
  // each quarter warp's sums (lanes 8g..8g+7); every lane of the warp takes part
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    r0.ss += __shfl_xor_sync(0xffffffffu, r0.ss, o);
    r1.ss += __shfl_xor_sync(0xffffffffu, r1.ss, o);
  }
  finish_row(p, r0, gl);
  finish_row(p, r1, gl);
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
  const int64_t rows_per_warp = kRowsPerQuarter * kRowsPerWarp;
  const int64_t warps_per_token = (num_q_heads + 2 * num_kv_heads + rows_per_warp - 1) / rows_per_warp;
  const int64_t warps = num_tokens * warps_per_token;
  const int64_t grid = (warps + kThreads / 32 - 1) / (kThreads / 32);
  if (grid * (kThreads / 32) > UINT32_MAX || grid > INT32_MAX) return PKV_ERR_UNSUPPORTED;
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
      prm, (uint32_t)warps_per_token);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
