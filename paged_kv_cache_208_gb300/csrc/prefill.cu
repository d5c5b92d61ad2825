// prefill.cu -- varlen causal prefill attention on the 5th-generation tensor cores (sm_103a).
//
// flash_attn_varlen_func of «nano-vLLM 最小化vLLM重新实现», 架构 5: causal attention over
// cu_seqlens-packed prompts, keys either packed or read from the paged pool through a block
// table (prefix caching, where queries cover only the uncached suffix and the causal mask is
// aligned to the end of the keys).
//
// Work unit (one CTA): sequence n, KV head h and a tile of 128 rows = the G query heads of h
// (G = Hq / Hkv) x 128/G consecutive query tokens, so every K/V tile loaded serves all G
// heads. For each 128-key tile j of the visible keys:
//   S_j = Q K_j^T   (tcgen05.mma, A = Q and B = K_j from shared memory, S_j in TMEM)
//   softmax warps: S_j row -> registers (tcgen05.ld), scale, causal mask, online max/sum in
//                  the log2 domain, P_j = 2^(s - m) as bf16 into shared memory
//   O += P_j V_j    (tcgen05.mma, A = P_j, B = V_j (MN-major), O accumulated in TMEM)
// O is rescaled in TMEM only when a row's running max grows by more than 2^8 (the sum l
// carries the same stale max, so O / l is unchanged).
//
// Warp roles (192 threads): warps 0-3 softmax + epilogue (thread = row = TMEM lane), warp 4
// TMA producer (Q once; K and V in 2-stage rings), warp 5 UMMA issuer and TMEM owner.
// TMEM columns: S double buffer [0, 256), O [256, 384).
// Shared memory: Q, 2 x K, 2 x V, P tiles of 32 KiB, all 128-byte swizzled, 1024-aligned.
//
// Rows of the last V tile past the sequence's keys are zeroed in shared memory before use
// (P is 0 there, but 0 x NaN from a stale pool slot would still poison O).
#include <math.h>

#include "device_common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace pkv {
namespace {

constexpr int kD = 128;
constexpr int kBM = 128;  // tile rows (G heads x 128/G tokens)
constexpr int kBN = 128;  // keys per tile
constexpr int kStages = 2;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 192;
constexpr uint32_t kTileBytes = kBM * kD * 2;  // 32 KiB
constexpr uint32_t kHalfBytes = kTileBytes / 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;

struct PrefillSmem {
  uint8_t q[kTileBytes];
  uint8_t k[kStages][kTileBytes];
  uint8_t v[kStages][kTileBytes];
  uint8_t p[kTileBytes];
  uint64_t q_full;
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t v_full[kStages], v_empty[kStages];
  uint64_t v_fixed;
  uint64_t s_full[2];
  uint64_t p_full;
  uint64_t o_full;
  uint32_t tmem_base;
};

struct PrefillParams {
  const int32_t *cu_q;
  const int32_t *cu_k;
  const int32_t *block_table;
  int32_t table_width;
  int32_t block_size;
  int64_t num_blocks;
  int64_t total_q;
  int64_t kv_rows;
  int32_t num_q_heads;
  int32_t qtiles;
  float scale_log2;
  int32_t causal;
  uint16_t *out;
  unsigned int *err;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
  constexpr int QT = kBM / G;  // query tokens per tile
  const int qt = p.qtiles - 1 - (int)blockIdx.x;  // longest (most keys) tiles first
  const int h = blockIdx.y;
  const int n = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int64_t q0 = p.cu_q[n], Lq = p.cu_q[n + 1] - q0;
  const int64_t k0 = p.cu_k[n], Lk = p.cu_k[n + 1] - k0;
  bool bad = Lq < 0 || Lk < 0 || q0 < 0 || q0 + Lq > p.total_q;
  if (p.block_table) bad = bad || Lk > (int64_t)p.table_width * p.block_size;
  else bad = bad || k0 < 0 || k0 + Lk > p.kv_rows;
  if (bad) {
    if (tid == 0 && qt == p.qtiles - 1 && h == 0) record_error(p.err, 8u /* SEQLEN_RANGE */);
    return;
  }
  if (tid == 0 && qt == p.qtiles - 1 && h == 0 && Lq > (int64_t)p.qtiles * QT)
    record_error(p.err, 8u);
  const int64_t qbeg = (int64_t)qt * QT;
  if (qbeg >= Lq) return;
  const int hq0 = h * G;
  const int64_t qlast = min(Lq, qbeg + QT) - 1;
  const int64_t kv_end = p.causal ? min(Lk, qlast + (Lk - Lq) + 1) : Lk;
  const int nk = kv_end > 0 ? (int)((kv_end + kBN - 1) / kBN) : 0;

  if (nk == 0) {  // no row of this tile sees a key: zeros
    for (int idx = tid; idx < kBM * 16; idx += kThreads) {
      const int r = idx >> 4, c = idx & 15;
      const int64_t qi = qbeg + r % QT;
      if (qi < Lq)
        reinterpret_cast<uint4 *>(p.out + ((q0 + qi) * p.num_q_heads + hq0 + r / QT) * kD)[c] =
            make_uint4(0, 0, 0, 0);
    }
    return;
  }
  // rows of the last key tile that hold keys of this sequence
  const int last_rows = (int)min((int64_t)kBN, Lk - (int64_t)(nk - 1) * kBN);
  const bool fix_v = last_rows < kBN;

  extern __shared__ uint8_t smem_raw[];
  PrefillSmem &sm = *reinterpret_cast<PrefillSmem *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  // an earlier wait gave up somewhere: return before allocating anything (uniform)
  if (__syncthreads_or(tid == 0 && aborted(p.err))) return;
  if (tid == 0) {
    mbar_init(&sm.q_full, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm.k_full[i], 1);
      mbar_init(&sm.k_empty[i], 1);
      mbar_init(&sm.v_full[i], 1);
      mbar_init(&sm.v_empty[i], 1);
      mbar_init(&sm.s_full[i], 1);
    }
    mbar_init(&sm.v_fixed, 1);
    mbar_init(&sm.p_full, 4);
    mbar_init(&sm.o_full, 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sm.tmem_base;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ TMA producer
    int issued = 0;
    bool ok = true;
    if (lane == 0) {
      prefetch_tensormap(&qmap);
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      mbar_arrive_expect_tx(&sm.q_full, kTileBytes);
      for (int g = 0; g < G; ++g)
        for (int hf = 0; hf < 2; ++hf)
          tma_load_3d(sm.q + hf * kHalfBytes + g * QT * 128, &qmap, &sm.q_full, 0,
                      (int32_t)(q0 + qbeg), 2 * (hq0 + g) + hf, pol_q);
      for (int j = 0; j < nk; ++j) {
        const int st = j % kStages;
        int32_t row;
        if (p.block_table) {
          const int64_t key = (int64_t)j * kBN;
          const int64_t blk = p.block_table[(int64_t)n * p.table_width + key / p.block_size];
          if (blk < 0 || blk >= p.num_blocks) {
            record_error(p.err, 2u /* BLOCK_RANGE */);
            row = -2 * kBN;  // wholly outside the pool: TMA fills zeros
          } else {
            row = (int32_t)(blk * p.block_size + key % p.block_size);
          }
        } else {
          row = (int32_t)(k0 + (int64_t)j * kBN);
        }
        if (j >= kStages && !wait_parity(&sm.k_empty[st], ((j / kStages) - 1) & 1, p.err)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&sm.k_full[st], kTileBytes);
        tma_load_3d(sm.k[st], &kmap, &sm.k_full[st], 0, row, 2 * h, pol_kv);
        if (j >= kStages && !wait_parity(&sm.v_empty[st], ((j / kStages) - 1) & 1, p.err)) {
          ok = false;
          issued = -(j + 1);  // K_j issued, V_j not
          break;
        }
        mbar_arrive_expect_tx(&sm.v_full[st], kTileBytes);
        tma_load_3d(sm.v[st], &vmap, &sm.v_full[st], 0, row, 2 * h, pol_kv);
        issued = j + 1;
      }
      if (!ok) record_error(p.err, 16u /* TIMEOUT */);
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (ok && fix_v) {
      const int j = nk - 1, st = j % kStages;
      const bool landed = wait_parity(&sm.v_full[st], (j / kStages) & 1, p.err);
      if (landed) {
        uint8_t *vt = sm.v[st];
        for (int idx = lane; idx < (kBN - last_rows) * 16; idx += 32) {
          const int r = last_rows + (idx >> 4), c = idx & 15;
          *reinterpret_cast<uint4 *>(vt + (c >> 3) * kHalfBytes + r * 128 + (c & 7) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_async_shared();
      } else if (lane == 0) {
        record_error(p.err, 16u);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.v_fixed);
    }
    if (lane == 0) {  // keep the CTA alive until every copy issued has landed
      const int kdone = issued >= 0 ? issued : -issued;
      const int vdone = issued >= 0 ? issued : -issued - 1;
      bool drained = wait_parity(&sm.q_full, 0, p.err);
      for (int j = max(0, kdone - kStages); drained && j < kdone; ++j)
        drained = wait_parity(&sm.k_full[j % kStages], (j / kStages) & 1, p.err);
      for (int j = max(0, vdone - kStages); drained && j < vdone; ++j)
        drained = wait_parity(&sm.v_full[j % kStages], (j / kStages) & 1, p.err);
      if (!drained) record_error(p.err, 16u);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ UMMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(kBM, kBN, 0, 0);  // Q (K-major) x K (K-major)
      constexpr uint32_t kIdO = idesc_bf16_f32(kBM, kD, 0, 1);   // P (K-major) x V (MN-major)
      const uint32_t qa = smem_addr(sm.q), pa = smem_addr(sm.p);
      bool ok = wait_parity(&sm.q_full, 0, p.err);
      auto issue_pv = [&](int i) {
        if (!ok) return;
        const int st = i % kStages;
        ok = wait_parity(&sm.p_full, i & 1, p.err) &&
             ((i == nk - 1 && fix_v) ? wait_parity(&sm.v_fixed, 0, p.err)
                                     : wait_parity(&sm.v_full[st], (i / kStages) & 1, p.err));
        if (!ok) return;
        tc_fence_after_sync();
        const uint32_t va = smem_addr(sm.v[st]);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t ad = smem_desc_sw128(pa + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(va + kk * 16 * 128, kHalfBytes, 1024);
          umma_bf16(tmem + kTmemO, ad, bd, kIdO, (i > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&sm.v_empty[st]);
        umma_commit(&sm.o_full);
      };
      for (int j = 0; j < nk && ok; ++j) {
        const int st = j % kStages;
        ok = wait_parity(&sm.k_full[st], (j / kStages) & 1, p.err);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t ka = smem_addr(sm.k[st]);
        const uint32_t d = tmem + (uint32_t)(j & 1) * kBN;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          umma_bf16(d, smem_desc_sw128(qa + off, 16, 1024), smem_desc_sw128(ka + off, 16, 1024),
                    kIdS, kk > 0 ? 1u : 0u);
        }
        umma_commit(&sm.k_empty[st]);
        umma_commit(&sm.s_full[j & 1]);
        if (j >= 1) issue_pv(j - 1);
      }
      issue_pv(nk - 1);
      // every UMMA must be complete before the tensor memory is released
      if (!ok || !wait_parity(&sm.o_full, (nk - 1) & 1, p.err)) record_error(p.err, 16u);
    }
  } else {
    // ------------------------------------------------------------------ softmax warps
    const int r = tid;  // tile row == TMEM lane
    const int g = r / QT;
    const int64_t qi = qbeg + r % QT;
    const bool row_valid = qi < Lq;
    int64_t lim = !row_valid ? -1 : (p.causal ? qi + (Lk - Lq) : Lk - 1);
    if (lim > Lk - 1) lim = Lk - 1;
    const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
    const int sw = r & 7;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nk; ++j) {
      // warp-uniform results: the TMEM loads and stores below are .sync.aligned
      if (!__all_sync(0xffffffffu, wait_parity(&sm.s_full[j & 1], (j >> 1) & 1, p.err))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      uint32_t s[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(lane_addr + (uint32_t)(j & 1) * kBN + c * 32, s[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_wait(s[c]);

      const int64_t kbase = (int64_t)j * kBN;
      const bool full = kbase + kBN - 1 <= lim;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float x = __uint_as_float(s[c][e]) * p.scale_log2;
          if (!full && kbase + c * 32 + e > lim) x = -INFINITY;
          s[c][e] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
      const float m_new = fmaxf(m_run, mx);
      const bool rescale = m_new > m_run + kRescaleLog2;
      float alpha = 1.f;
      if (rescale) {
        alpha = fast_exp2(m_run - m_new);
        m_run = m_new;
        l_run *= alpha;
      }
      const float m_use = m_run == -INFINITY ? 0.f : m_run;
      uint32_t pk[64];
      float rowsum = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = fast_exp2(__uint_as_float(s[c][2 * e]) - m_use);
          const float p1 = fast_exp2(__uint_as_float(s[c][2 * e + 1]) - m_use);
          rowsum += p0 + p1;
          pk[c * 16 + e] = pack_bf16(p0, p1);
        }
      l_run += rowsum;

      // P_{j-1} V_{j-1} must be done before P is overwritten and O is rescaled
      if (j >= 1) {
        if (!__all_sync(0xffffffffu, wait_parity(&sm.o_full, (j - 1) & 1, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
      }
#pragma unroll
      for (int c16 = 0; c16 < 16; ++c16) {
        uint8_t *dst = sm.p + (c16 >> 3) * kHalfBytes + r * 128 + (((c16 & 7) ^ sw) << 4);
        *reinterpret_cast<uint4 *>(dst) =
            make_uint4(pk[4 * c16], pk[4 * c16 + 1], pk[4 * c16 + 2], pk[4 * c16 + 3]);
      }
      if (j >= 1 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(lane_addr + kTmemO + c * 32, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(lane_addr + kTmemO + c * 32, o);
        }
        tmem_st_wait();
      }
      fence_async_shared();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_full);
    }
    // ---- epilogue: O / l -> bf16 rows
    if (ok) ok = __all_sync(0xffffffffu, wait_parity(&sm.o_full, (nk - 1) & 1, p.err));
    if (ok) {
      tc_fence_after_sync();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      uint4 *dst = reinterpret_cast<uint4 *>(p.out + ((q0 + qi) * p.num_q_heads + hq0 + g) * kD);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(lane_addr + kTmemO + c * 32, o);
        tmem_ld_wait(o);
        if (row_valid) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 v4;
            v4.x = pack_bf16(__uint_as_float(o[8 * e + 0]) * inv, __uint_as_float(o[8 * e + 1]) * inv);
            v4.y = pack_bf16(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv);
            v4.z = pack_bf16(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv);
            v4.w = pack_bf16(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv);
            dst[c * 4 + e] = v4;
          }
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int G>
cudaError_t launch_g(const PrefillArgs &a, const PrefillParams &prm, cudaStream_t stream) {
  constexpr int QT = kBM / G;
  CUtensorMap qm, km, vm;
  const uint64_t qdims[3] = {64, (uint64_t)a.total_q, (uint64_t)a.num_q_heads * 2};
  const uint64_t qstr[2] = {(uint64_t)a.q_tok_stride * 2, 128};
  const uint32_t qbox[3] = {64, (uint32_t)QT, 1};
  const uint64_t kvdims[3] = {64, (uint64_t)(a.kv_rows > 0 ? a.kv_rows : 1),
                              (uint64_t)a.num_kv_heads * 2};
  const uint64_t kvstr[2] = {(uint64_t)a.kv_tok_stride * 2, 128};
  const uint32_t kvbox[3] = {64, (uint32_t)kBN, 2};
  if (encode_tensor_map(&qm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.q), qdims,
                        qstr, qbox, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B) != CUDA_SUCCESS ||
      encode_tensor_map(&km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.k), kvdims,
                        kvstr, kvbox, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B) != CUDA_SUCCESS ||
      encode_tensor_map(&vm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.v), kvdims,
                        kvstr, kvbox, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(PrefillSmem) + 1024;
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  PrefillParams p2 = prm;
  p2.qtiles = (a.max_seqlen_q + QT - 1) / QT;
  const dim3 grid((unsigned)p2.qtiles, (unsigned)a.num_kv_heads, (unsigned)a.num_seqs);
  prefill_kernel<G><<<grid, kThreads, smem, stream>>>(qm, km, vm, p2);
  return cudaGetLastError();
}

}  // namespace

bool prefill_group_supported(int group) {
  return group == 1 || group == 2 || group == 4 || group == 8;
}

cudaError_t launch_varlen_prefill(const PrefillArgs &a, int num_sms, cudaStream_t stream) {
  (void)num_sms;
  PrefillParams prm{};
  prm.cu_q = a.cu_seqlens_q;
  prm.cu_k = a.cu_seqlens_k;
  prm.block_table = a.block_table;
  prm.table_width = a.table_width;
  prm.block_size = a.block_size;
  prm.num_blocks = a.num_blocks;
  prm.total_q = a.total_q;
  prm.kv_rows = a.kv_rows;
  prm.num_q_heads = a.num_q_heads;
  prm.scale_log2 = a.scale * kLog2e;
  prm.causal = a.causal;
  prm.out = static_cast<uint16_t *>(a.out);
  prm.err = a.err;
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_g<1>(a, prm, stream);
    case 2: return launch_g<2>(a, prm, stream);
    case 4: return launch_g<4>(a, prm, stream);
    case 8: return launch_g<8>(a, prm, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace pkv
