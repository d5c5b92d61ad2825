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
// A warp owns one token. Its lane 0 brings the whole projection row (contiguous, 8 KiB for
// 16 + 2 x 8 heads) into shared memory with one 1-D bulk copy, so a CTA keeps eight rows in
// flight with no registers held for them. The warp then normalises and rotates the query and
// key heads in place, eight rows at a time: a quarter warp (8 lanes) owns a head row, lane l
// holding elements 8l..8l+7 and their RoPE partners 64+8l..64+8l+7, so the rotation needs no
// exchange and the sum of squares takes three shuffles. Lane 0 then writes the token's q
// heads, K heads and (untouched) V heads out with three bulk copies: q_out[t], and the
// pool rows of slot[t]. Roundings to bf16 go two values per conversion instruction.
#include <math.h>

#include <algorithm>
#include <stdint.h>

#include <cuda_bf16.h>

#include "device_common.cuh"
#include "launch.h"
#include "pkv.h"

namespace pkv {
namespace {

constexpr int kD = 128;
constexpr int kHalf = kD / 2;
constexpr int kRowBytes = kD * 2;     // one head row, bf16
constexpr int kMaxTokensPerCta = 8;   // one warp per token
constexpr int kMaxSmem = 96 * 1024;   // staged projection rows per CTA (two CTAs per SM)

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

__device__ __forceinline__ float sum_sq(const uint4 lo, const uint4 hi) {
  float a[8], b[8];
  unpack8(lo, a);
  unpack8(hi, b);
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) ss = fmaf(a[i], a[i], fmaf(b[i], b[i], ss));
  return ss;
}

// Normalise and rotate one head row held by a quarter warp (lo, hi: this lane's 8 + 8
// elements), once its sum of squares is known; the result goes back over the row.
__device__ __forceinline__ void finish_row(const RopeParams &p, uint8_t *row, uint4 lo, uint4 hi,
                                           float ss, bool is_q, const float4 (&cs)[4], int gl) {
  const float rs = rsqrtf(ss * (1.f / kD) + p.eps);
  const uint16_t *wsrc = is_q ? p.q_weight : p.k_weight;
  float a[8], b[8], wa[8], wb[8];
  unpack8(lo, a);
  unpack8(hi, b);
  unpack8(*reinterpret_cast<const uint4 *>(wsrc + 8 * gl), wa);
  unpack8(*reinterpret_cast<const uint4 *>(wsrc + kHalf + 8 * gl), wb);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    a[i] = a[i] * rs * wa[i];
    b[i] = b[i] * rs * wb[i];
  }
  round8(a);
  round8(b);
  const float c[8] = {cs[0].x, cs[0].y, cs[0].z, cs[0].w, cs[1].x, cs[1].y, cs[1].z, cs[1].w};
  const float s[8] = {cs[2].x, cs[2].y, cs[2].z, cs[2].w, cs[3].x, cs[3].y, cs[3].z, cs[3].w};
  float ya[8], yb[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    ya[i] = a[i] * c[i] - b[i] * s[i];
    yb[i] = b[i] * c[i] + a[i] * s[i];
  }
  reinterpret_cast<uint4 *>(row)[gl] = pack8(ya);
  reinterpret_cast<uint4 *>(row + kHalf * 2)[gl] = pack8(yb);
}

__global__ void __launch_bounds__(kMaxTokensPerCta * 32)
    qk_norm_rope_store_kernel(const RopeParams p, int tokens_per_cta) {
  extern __shared__ __align__(128) uint8_t rows[];  // tokens_per_cta staged projection rows
  __shared__ uint64_t row_full[kMaxTokensPerCta];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int group = lane >> 3, gl = lane & 7;
  const int heads = p.hq + 2 * p.hkv;
  const uint32_t row_bytes = (uint32_t)heads * kRowBytes;
  if (threadIdx.x == 0) {
    for (int i = 0; i < tokens_per_cta; ++i) mbar_init(&row_full[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int64_t t = (int64_t)blockIdx.x * tokens_per_cta + warp;
  if (warp >= tokens_per_cta || t >= p.num_tokens) return;
  // an earlier wait gave up somewhere: issue nothing (warp-uniform)
  if (__any_sync(0xffffffffu, lane == 0 && aborted(p.err))) return;
  uint8_t *row = rows + (size_t)warp * row_bytes;
  if (lane == 0) {
    mbar_arrive_expect_tx(&row_full[warp], row_bytes);
    bulk_copy_g2s(row, p.qkv + t * p.tok_stride, row_bytes, &row_full[warp]);
  }
  // while the row is in flight: this token's position, slot and cos/sin
  const int64_t pos = p.positions[t];
  const int64_t slot = p.slots[t];
  const bool pos_ok = pos >= 0 && pos < p.max_position;
  const bool slot_ok = slot >= 0 && slot < p.num_slots;
  if (lane == 0) {
    if (!pos_ok) record_error(p.err, 32u /* POSITION_RANGE */);
    if (slot >= p.num_slots) record_error(p.err, 1u /* SLOT_RANGE */);
  }
  float4 cs[4] = {};
  if (pos_ok) {
    const float4 *src = reinterpret_cast<const float4 *>(p.cos_sin + pos * kD);
    cs[0] = src[2 * gl];
    cs[1] = src[2 * gl + 1];
    cs[2] = src[16 + 2 * gl];
    cs[3] = src[16 + 2 * gl + 1];
  }
  // the warp's own copy: wait for it to land even if another CTA has given up meanwhile
  if (!__all_sync(0xffffffffu, wait_own(&row_full[warp], 0, p.err))) return;
  if (pos_ok) {
    // query and key heads, eight rows per pass (two per quarter warp); every lane takes part
    // in the shuffles, rows past the key heads contribute zeros
    const int nqk = p.hq + p.hkv;
    for (int h0 = 0; h0 < nqk; h0 += 8) {
      const int ha = h0 + group, hb = h0 + 4 + group;
      uint8_t *ra = row + (size_t)ha * kRowBytes, *rb = row + (size_t)hb * kRowBytes;
      const uint4 z = make_uint4(0, 0, 0, 0);
      const uint4 alo = ha < nqk ? reinterpret_cast<const uint4 *>(ra)[gl] : z;
      const uint4 ahi = ha < nqk ? reinterpret_cast<const uint4 *>(ra + kHalf * 2)[gl] : z;
      const uint4 blo = hb < nqk ? reinterpret_cast<const uint4 *>(rb)[gl] : z;
      const uint4 bhi = hb < nqk ? reinterpret_cast<const uint4 *>(rb + kHalf * 2)[gl] : z;
      float sa = sum_sq(alo, ahi), sb = sum_sq(blo, bhi);
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {
        sa += __shfl_xor_sync(0xffffffffu, sa, o);
        sb += __shfl_xor_sync(0xffffffffu, sb, o);
      }
      if (ha < nqk) finish_row(p, ra, alo, ahi, sa, ha < p.hq, cs, gl);
      if (hb < nqk) finish_row(p, rb, blo, bhi, sb, hb < p.hq, cs, gl);
    }
    fence_async_shared();  // the rows written above are read by the bulk copies below
  }
  __syncwarp();
  if (lane == 0) {
    const uint32_t q_bytes = (uint32_t)p.hq * kRowBytes, kv_bytes = (uint32_t)p.hkv * kRowBytes;
    if (pos_ok) bulk_copy_s2g(p.q_out + t * p.hq * kD, row, q_bytes);
    if (slot_ok) {
      if (pos_ok) bulk_copy_s2g(p.k_cache + slot * p.hkv * kD, row + q_bytes, kv_bytes);
      bulk_copy_s2g(p.v_cache + slot * p.hkv * kD, row + q_bytes + kv_bytes, kv_bytes);
    }
    bulk_commit();
    bulk_wait_read_all();  // the row must stay in shared memory until the copies have read it
  }
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
  const int64_t row_bytes = (int64_t)(num_q_heads + 2 * num_kv_heads) * head_dim * 2;
  const int64_t tpc = row_bytes > kMaxSmem ? 1 : std::min<int64_t>(kMaxTokensPerCta, kMaxSmem / row_bytes);
  const int64_t smem = tpc * row_bytes;
  const int64_t grid = (num_tokens + tpc - 1) / tpc;
  if (grid > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  // once per device: allow dynamic shared memory up to the per-CTA maximum
  static int max_dynamic[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  int limit = dev < 64 ? max_dynamic[dev] : 0;
  if (limit == 0) {
    int optin = 0;
    cudaFuncAttributes fa{};
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        cudaFuncGetAttributes(&fa, qk_norm_rope_store_kernel) != cudaSuccess)
      return PKV_ERR_CUDA;
    limit = optin - (int)fa.sharedSizeBytes;
    if (cudaFuncSetAttribute(qk_norm_rope_store_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, limit) != cudaSuccess)
      return PKV_ERR_CUDA;
    if (dev < 64) max_dynamic[dev] = limit;
  }
  if (smem > limit) return PKV_ERR_UNSUPPORTED;  // one token's row does not fit
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
  qk_norm_rope_store_kernel<<<(unsigned)grid, (unsigned)(tpc * 32), (size_t)smem,
                              static_cast<cudaStream_t>(stream)>>>(prm, (int)tpc);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
