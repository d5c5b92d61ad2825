// prefill.cu -- varlen causal prefill attention on the 5th-generation tensor cores (sm_103a).
//
// flash_attn_varlen_func of «nano-vLLM 最小化vLLM重新实现», 架构 5: causal attention over
// cu_seqlens-packed prompts, keys either packed or read from the paged pool through a block
// table (prefix caching: queries cover only the uncached suffix and the causal mask is
// aligned to the end of the keys).
//
// Persistent kernel: one CTA per SM takes work items from a global queue (an atomic counter
// in the caller's workspace). A one-CTA planning kernel first writes the work list there:
// only (sequence, query block) units that have queries, sequences with the most query blocks
// first and each sequence's blocks heaviest first, all heads of a unit next to each other.
// The heavy work starts first (the queue balances the SMs), and the query blocks of one
// sequence run at about the same time, so the K/V tiles they share come from L2. The
// producer warp takes the items and hands them to the other warps through a small ring in
// shared memory. An item is
// one sequence n, one KV head h and two 128-row M-tiles that share every K/V tile: for a GQA
// group of two (or a pair of heads of a larger group) the two query heads over the same 128
// tokens; without GQA two consecutive 128-token blocks of the one head. Per 128-key tile j:
//   S_a = Q_a K_j^T      tcgen05.mma, Q_a and K_j from shared memory, S_a in TMEM
//   softmax warpgroup a  row max (pass 1) and P_a = 2^(s - m) (pass 2) read from TMEM with
//                        tcgen05.ld; P_a written back as bf16 over S_a's first 64 columns
//   O_a += P_a V_j        tcgen05.mma with A = P_a read from TMEM, B = V_j (MN-major) in smem
// The MMA warp issues S_0(j), O_1 += P_1(j-1) V(j-1), S_1(j), O_0 += P_0(j) V(j), so each
// softmax warpgroup works while the tensor core serves the other. O_a is rescaled in TMEM
// only when a row's running max grows by more than 2^8 (its sum l carries the same stale
// max, so O / l is unchanged).
//
// Warps (384 threads): 0-3 softmax/epilogue of M-tile 0, 4-7 of M-tile 1 (thread = row =
// TMEM lane), 8 scheduler + TMA producer (Q_0, Q_1 per item, each reloaded as soon as its
// last S MMA is done; K and V tiles through one 5-slot ring), 9 UMMA issuer and TMEM
// owner, 10-11 idle. TMEM: S_0 [0,128), S_1 [128,256), O_0 [256,384),
// O_1 [384,512). Shared memory: Q_0, Q_1 and 5 K/V slots of 32 KiB, 128-byte swizzled.
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
constexpr int kBM = 128;  // rows of one M-tile
constexpr int kBN = 128;  // keys per tile
constexpr int kSlots = 5;  // K/V ring: K(j) is load 2j and V(j) load 2j + 1, slot = load % 5
constexpr int kThreads = 384;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTileBytes = kBM * kD * 2;  // 32 KiB
constexpr uint32_t kHalfBytes = kTileBytes / 2;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;
constexpr unsigned kFull = 0xffffffffu;
// Registers per thread: at launch (= 65536 / 384, what __launch_bounds__(384, 1) gives) and
// after the split. 2 x kSoftmaxRegs + kOtherRegs must not exceed 3 x kLaunchRegs, or the
// increase would wait forever; the launcher checks the compiled count before every launch.
constexpr int kLaunchRegs = 168;
constexpr int kSoftmaxRegs = 208;
constexpr int kOtherRegs = 88;
static_assert(2 * kSoftmaxRegs + kOtherRegs <= 3 * kLaunchRegs, "register split too large");

template <int N>
__device__ __forceinline__ void reg_alloc_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void reg_dealloc() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

struct Item {
  int id;          // index in the work list; -1 marks the end of the work
  int n, h;
  int hq[2];
  int64_t tok[2];  // first query token (within the sequence) of each M-tile
  int64_t q0, Lq, k0, Lk;
  int nk;          // key tiles to process
  int last_rows;   // keys of the sequence in the last key tile
  bool valid;      // the item has queries
  bool bad;        // cu_seqlens / block_table inconsistent for this sequence
};

constexpr int kRing = 4;  // work items in flight between the scheduler and the other warps

struct PrefillSmem {
  uint8_t q[2][kTileBytes];
  uint8_t kv[kSlots][kTileBytes];
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full[kSlots], kv_empty[kSlots];
  uint64_t v_fixed[kSlots];  // per slot: the next fix of a slot needs that slot released
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t mma_drain;  // the MMA thread's last commit: every UMMA it issued has completed
  uint64_t item_full[kRing], item_empty[kRing];
  Item items[kRing];  // decoded once by the scheduler, read by the other warps
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
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  const int2 *units;        // work list: (sequence, query block), written by the planner
  const int32_t *num_units; // its length (written by the planner)
  float scale_log2;
  int32_t causal;
  uint16_t *out;
  bool out_32b;    // out is 32-byte aligned: rows are written with 32-byte stores
  int32_t *queue;  // next item to hand out (zeroed before the launch)
  unsigned int *err;
};


// Item i of the work list: unit i / (KV heads x head pairs), head pair i % that.
template <int G>
__device__ __forceinline__ Item decode_item(const PrefillParams &p, int i) {
  constexpr int kPairs = G >= 2 ? G / 2 : 1;
  Item it;
  it.id = i;
  const int per_unit = p.num_kv_heads * kPairs;
  const int2 u = p.units[i / per_unit];
  const int hp = i % per_unit;
  const int qb = u.y;
  it.n = u.x;
  it.h = hp / kPairs;
  const int pair = hp % kPairs;
  if (G >= 2) {
    it.hq[0] = it.h * G + 2 * pair;
    it.hq[1] = it.hq[0] + 1;
    it.tok[0] = it.tok[1] = (int64_t)qb * kBM;
  } else {
    it.hq[0] = it.hq[1] = it.h;
    it.tok[0] = (int64_t)qb * 2 * kBM;
    it.tok[1] = it.tok[0] + kBM;
  }
  it.q0 = p.cu_q[it.n];
  it.Lq = p.cu_q[it.n + 1] - it.q0;
  it.k0 = p.cu_k[it.n];
  it.Lk = p.cu_k[it.n + 1] - it.k0;
  bool bad = it.Lq < 0 || it.Lk < 0 || it.q0 < 0 || it.q0 + it.Lq > p.total_q;
  if (p.block_table) bad = bad || it.Lk > (int64_t)p.table_width * p.block_size;
  else bad = bad || it.k0 < 0 || it.k0 + it.Lk > p.kv_rows;
  it.bad = bad;
  it.valid = !bad && it.tok[0] < it.Lq;
  it.nk = 0;
  it.last_rows = 0;
  if (it.valid) {
    int64_t kv_end = 0;
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      if (it.tok[a] >= it.Lq) continue;
      const int64_t last_q = min(it.Lq, it.tok[a] + kBM) - 1;
      const int64_t e = p.causal ? min(it.Lk, last_q + (it.Lk - it.Lq) + 1) : it.Lk;
      kv_end = max(kv_end, e);
    }
    if (kv_end > 0) {
      it.nk = (int)((kv_end + kBN - 1) / kBN);
      it.last_rows = (int)min((int64_t)kBN, it.Lk - (int64_t)(it.nk - 1) * kBN);
    }
  }
  return it;
}

// Next work item from the ring (in order), taken by a whole warp: every lane waits, and the
// item counts only if every lane saw it (so the warp agrees even when a wait gives up).
// Returns the slot, or nullptr when the wait gave up. The caller reads the fields it needs
// in place and then releases the slot (release_item).
__device__ __forceinline__ const Item *wait_item(PrefillSmem &sm, uint32_t taken,
                                                 unsigned int *err) {
  const int slot = taken % kRing;
  if (__all_sync(0xffffffffu, wait_parity(&sm.item_full[slot], (taken / kRing) & 1, err)))
    return &sm.items[slot];
  return nullptr;
}

__device__ __forceinline__ void release_item(PrefillSmem &sm, uint32_t taken, int lane) {
  __syncwarp();  // every lane has read the item before the slot is released
  if (lane == 0) mbar_arrive(&sm.item_empty[taken % kRing]);
}

// S = Q K^T for one 128 x 128 tile: 8 UMMAs of K = 16 over the two 64-column halves. The
// descriptors are the tiles' base descriptors plus compile-time offsets (the start address
// sits in the low bits, in 16-byte units). Called by the whole MMA warp; one lane issues.
__device__ __forceinline__ void mma_qk(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc,
                                       uint32_t idesc) {
  if (elect_one()) {
    umma_ss<false>(d_tmem, q_desc, k_desc, idesc);
#pragma unroll
    for (int kk = 1; kk < kD / 16; ++kk) {
      const uint64_t off = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
      umma_ss<true>(d_tmem, q_desc + off, k_desc + off, idesc);
    }
  }
  __syncwarp();
}

// O (+)= P V for one tile: P from TMEM (8 columns per 16 keys), V MN-major in smem (16 keys
// = 2 KiB further per step).
__device__ __forceinline__ void mma_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t v_desc,
                                       uint32_t idesc, bool accumulate) {
  if (elect_one()) {
    if (accumulate) umma_ts<true>(d_tmem, p_tmem, v_desc, idesc);
    else umma_ts<false>(d_tmem, p_tmem, v_desc, idesc);
#pragma unroll
    for (int kk = 1; kk < kBN / 16; ++kk)
      umma_ts<true>(d_tmem, p_tmem + 8 * kk, v_desc + ((kk * 16 * 128) >> 4), idesc);
  }
  __syncwarp();
}

// tcgen05.commit from the lane that issued the UMMAs (the warp is converged here too).
__device__ __forceinline__ void commit_one(uint64_t *bar) {
  if (elect_one()) umma_commit(bar);
  __syncwarp();
}

// One 32-byte global store (sm_100 and later); p must be 32-byte aligned.
__device__ __forceinline__ void st_global_32b(void *p, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  extern __shared__ uint8_t smem_raw[];
  PrefillSmem &sm = *reinterpret_cast<PrefillSmem *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  // an earlier wait gave up somewhere: return before allocating anything (uniform)
  if (__syncthreads_or(tid == 0 && aborted(p.err))) return;
  if (tid == 0) {
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sm.q_full[a], 1);
      mbar_init(&sm.q_empty[a], 1);
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&sm.item_full[i], 1);
      mbar_init(&sm.item_empty[i], 1 + 8);  // the MMA thread and the 8 softmax warps
    }
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&sm.kv_full[i], 1);
      mbar_init(&sm.kv_empty[i], 1);
      mbar_init(&sm.v_fixed[i], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sm.s_full[a], 1);
      mbar_init(&sm.p_full[a], 4);
      mbar_init(&sm.o_full[a], 1);
    }
    mbar_init(&sm.mma_drain, 1);
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

  // Register split (launch: kLaunchRegs x 384 threads): the two softmax warpgroups hold a
  // whole 128-column S row per thread; warpgroup 2 only schedules, loads and issues MMAs.
  // Each warpgroup executes one setmaxnreg, and the roles are nested under it.
  if (warp >= 8) {
  reg_dealloc<kOtherRegs>();
  if (warp == kProducerWarp) {
    // ------------------------------------------------------------- scheduler + TMA producer
    uint64_t pol_q = 0, pol_kv = 0;
    if (lane == 0) {
      prefetch_tensormap(&qmap);
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
      pol_q = policy_evict_first();
      pol_kv = policy_evict_last();
    }
    uint32_t pushed = 0, q_loads = 0, g = 0;
    uint32_t q_issued[2] = {0, 0};  // loads issued into each Q buffer (lane 0's count)
    int last_load = -1;
    bool ok = true;
    const int total_items = lane == 0 ? *p.num_units * p.num_kv_heads * (G >= 2 ? G / 2 : 1) : 0;
    while (ok) {
      // take the next item that has queries; -1 when the queue is exhausted
      int i = -1;
      if (lane == 0) {
        Item d;
        d.id = -1;
        while (true) {
          i = atomicAdd(p.queue, 1);
          if (i >= total_items) break;
          d = decode_item<G>(p, i);
          if (d.bad) record_error(p.err, 8u /* SEQLEN_RANGE */);
          if (d.valid) break;
        }
        if (i >= total_items) {
          i = -1;
          d.id = -1;
        }
        const int slot = pushed % kRing;
        if (pushed >= kRing)
          ok = wait_parity(&sm.item_empty[slot], ((pushed / kRing) - 1) & 1, p.err);
        if (ok) {
          sm.items[slot] = d;
          mbar_arrive(&sm.item_full[slot]);  // release: the item is visible to the waiters
        }
      }
      ++pushed;
      ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
      i = __shfl_sync(kFull, i, 0);
      if (!ok || i < 0) break;
      __syncwarp();  // lane 0 wrote the slot
      const Item it = sm.items[(pushed - 1) % kRing];
      if (it.nk == 0) continue;  // no key visible: the softmax warps write zeros
      if (lane == 0) {
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          if (q_loads > 0) ok = ok && wait_parity(&sm.q_empty[a], (q_loads - 1) & 1, p.err);
          if (ok) {
            mbar_arrive_expect_tx(&sm.q_full[a], kTileBytes);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
              tma_load_3d(sm.q[a] + hf * kHalfBytes, &qmap, &sm.q_full[a], 0,
                          (int32_t)(it.q0 + it.tok[a]), 2 * it.hq[a] + hf, pol_q);
            ++q_issued[a];
          }
        }
      }
      ++q_loads;
      ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
      for (int j = 0; j < it.nk && ok; ++j, ++g) {
        const uint32_t nk_load = 2 * g, nv_load = 2 * g + 1;
        const int ks = nk_load % kSlots, vs = nv_load % kSlots;
        if (lane == 0) {
          int32_t row;
          if (p.block_table) {
            const int64_t key = (int64_t)j * kBN;
            const int64_t blk = p.block_table[(int64_t)it.n * p.table_width + key / p.block_size];
            if (blk < 0 || blk >= p.num_blocks) {
              record_error(p.err, 2u /* BLOCK_RANGE */);
              row = -2 * kBN;  // wholly outside the pool: TMA fills zeros
            } else {
              row = (int32_t)(blk * p.block_size + key % p.block_size);
            }
          } else {
            row = (int32_t)(it.k0 + (int64_t)j * kBN);
          }
          if (nk_load >= kSlots)
            ok = wait_parity(&sm.kv_empty[ks], ((nk_load / kSlots) - 1) & 1, p.err);
          if (ok) {
            mbar_arrive_expect_tx(&sm.kv_full[ks], kTileBytes);
            tma_load_3d(sm.kv[ks], &kmap, &sm.kv_full[ks], 0, row, 2 * it.h, pol_kv);
            last_load = (int)nk_load;
          }
          if (ok && nv_load >= kSlots)
            ok = wait_parity(&sm.kv_empty[vs], ((nv_load / kSlots) - 1) & 1, p.err);
          if (ok) {
            mbar_arrive_expect_tx(&sm.kv_full[vs], kTileBytes);
            tma_load_3d(sm.kv[vs], &vmap, &sm.kv_full[vs], 0, row, 2 * it.h, pol_kv);
            last_load = (int)nv_load;
          }
        }
        ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
        if (ok && j == it.nk - 1 && it.last_rows < kBN) {
          // zero the rows past the sequence's keys before the MMA reads this V tile
          ok = __all_sync(kFull, wait_parity(&sm.kv_full[vs], (nv_load / kSlots) & 1, p.err));
          if (ok) {
            uint8_t *vt = sm.kv[vs];
            for (int idx = lane; idx < (kBN - it.last_rows) * 16; idx += 32) {
              const int r = it.last_rows + (idx >> 4), c = idx & 15;
              *reinterpret_cast<uint4 *>(vt + (c >> 3) * kHalfBytes + r * 128 + (c & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            fence_async_shared();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.v_fixed[vs]);
          }
        }
      }
    }
    if (lane == 0) {
      // keep the CTA alive until every copy issued has landed, also after an abort (these
      // waits ignore the abort bit; only issued loads are waited for: each Q buffer's last
      // one, and the K/V loads up to last_load, which were issued in order)
      bool drained = true;
      for (int a = 0; a < 2; ++a)
        if (q_issued[a] > 0)
          drained = drained && wait_own(&sm.q_full[a], (q_issued[a] - 1) & 1, p.err);
      for (int t = max(0, last_load - kSlots + 1); drained && t <= last_load; ++t)
        drained = wait_own(&sm.kv_full[t % kSlots], (t / kSlots) & 1, p.err);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ UMMA issuer
    // The whole warp runs this loop (waits, descriptor arithmetic) so that it stays
    // converged; one elected lane issues each group of UMMAs and its commits.
    constexpr uint32_t kIdS = idesc_bf16_f32(kBM, kBN, 0, 0);  // Q (K-major) x K (K-major)
    constexpr uint32_t kIdO = idesc_bf16_f32(kBM, kD, 0, 1);   // P (TMEM) x V (MN-major)
    constexpr uint64_t kSlotStep = kTileBytes >> 4;            // one ring slot, descriptor units
    const uint64_t dq0 = smem_desc_sw128(smem_addr(sm.q[0]), 16, 1024);
    const uint64_t dq1 = smem_desc_sw128(smem_addr(sm.q[1]), 16, 1024);
    const uint64_t dk0 = smem_desc_sw128(smem_addr(sm.kv[0]), 16, 1024);
    const uint64_t dv0 = smem_desc_sw128(smem_addr(sm.kv[0]), kHalfBytes, 1024);
    uint32_t taken = 0, q_loads = 0, g = 0;
    uint32_t fix_parity = 0;  // bit s: parity of the next v_fixed phase of slot s
    bool ok = true;
    // warp-uniform wait
    auto wait_all = [&](uint64_t *bar, uint32_t parity) -> bool {
      return __all_sync(kFull, wait_parity(bar, parity, p.err));
    };
    // V(j) of tile gg: wait for the load (or, for a fixed last tile, for the fix)
    auto v_ready = [&](uint32_t gg, bool fixed) -> bool {
      const uint32_t n = 2 * gg + 1, vs = n % kSlots;
      if (fixed) {
        const bool r = wait_all(&sm.v_fixed[vs], (fix_parity >> vs) & 1);
        fix_parity ^= 1u << vs;
        return r;
      }
      return wait_all(&sm.kv_full[vs], (n / kSlots) & 1);
    };
    while (ok) {
      const Item *ip = wait_item(sm, taken, p.err);
      const int id = ip ? ip->id : -1, nk = ip ? ip->nk : 0;
      const bool fix_v = ip && ip->last_rows < kBN;
      release_item(sm, taken, lane);
      ++taken;
      if (id < 0) break;
      if (nk == 0) continue;
      for (int j = 0; j < nk; ++j, ++g) {
        const uint32_t ks = (2 * g) % kSlots;
        ok = wait_all(&sm.kv_full[ks], ((2 * g) / kSlots) & 1);
        if (!ok) break;
        tc_fence_after_sync();
        // S_0(j)
        if (j == 0) {
          ok = wait_all(&sm.q_full[0], q_loads & 1);
          if (!ok) break;
          tc_fence_after_sync();
        }
        mma_qk(tmem, dq0, dk0 + ks * kSlotStep, kIdS);
        commit_one(&sm.s_full[0]);
        if (j == nk - 1) commit_one(&sm.q_empty[0]);
        // O_1 += P_1(j-1) V(j-1)  (never the last tile here)
        if (j > 0) {
          const uint32_t gp = g - 1, vs = (2 * gp + 1) % kSlots;
          ok = wait_all(&sm.p_full[1], gp & 1) && v_ready(gp, false);
          if (!ok) break;
          tc_fence_after_sync();
          mma_pv(tmem + 384, tmem + 128, dv0 + vs * kSlotStep, kIdO, j - 1 > 0);
          commit_one(&sm.o_full[1]);
          commit_one(&sm.kv_empty[vs]);
        }
        // S_1(j)
        if (j == 0) {
          ok = wait_all(&sm.q_full[1], q_loads & 1);
          if (!ok) break;
          tc_fence_after_sync();
        }
        mma_qk(tmem + 128, dq1, dk0 + ks * kSlotStep, kIdS);
        commit_one(&sm.s_full[1]);
        if (j == nk - 1) commit_one(&sm.q_empty[1]);
        commit_one(&sm.kv_empty[ks]);
        // O_0 += P_0(j) V(j); for a fixed last tile this wait also covers O_1's use below
        ok = wait_all(&sm.p_full[0], g & 1) && v_ready(g, j == nk - 1 && fix_v);
        if (!ok) break;
        tc_fence_after_sync();
        mma_pv(tmem + 256, tmem, dv0 + ((2 * g + 1) % kSlots) * kSlotStep, kIdO, j > 0);
        commit_one(&sm.o_full[0]);
      }
      if (!ok) break;
      {  // O_1 += P_1(last) V(last): V(last) is ready (waited above)
        const uint32_t gp = g - 1, vs = (2 * gp + 1) % kSlots;
        ok = wait_all(&sm.p_full[1], gp & 1);
        if (!ok) break;
        tc_fence_after_sync();
        mma_pv(tmem + 384, tmem + 128, dv0 + vs * kSlotStep, kIdO, nk > 1);
        commit_one(&sm.o_full[1]);
        commit_one(&sm.kv_empty[vs]);
      }
      ++q_loads;
    }
    // every UMMA must be complete before the tensor memory is released and the CTA exits,
    // also after an abort: one more commit tracks all of them (the wait ignores the abort bit)
    commit_one(&sm.mma_drain);
    __all_sync(kFull, wait_own(&sm.mma_drain, 0, p.err));
  }
  } else {
    reg_alloc_inc<kSoftmaxRegs>();
    // ------------------------------------------------------------------ softmax warps
    const int a = warp >> 2;        // M-tile
    const int r = tid & (kBM - 1);  // row == TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t s_col = 128 * a, o_col = 256 + 128 * a;
    const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
    uint32_t taken = 0, g = 0;
    bool ok = true;
    while (ok) {
      const Item *ip = wait_item(sm, taken, p.err);
      const int id = ip ? ip->id : -1, nk = ip ? ip->nk : 0;
      int64_t row = -1;  // output row (token x head) of this thread; -1 past the queries
      int64_t lim = -1;  // last key this row sees (-1: none)
      if (id >= 0) {
        const int64_t qi = ip->tok[a] + r, Lq = ip->Lq, Lk = ip->Lk;
        if (qi < Lq) {
          row = (ip->q0 + qi) * p.num_q_heads + ip->hq[a];
          lim = min(p.causal ? qi + (Lk - Lq) : Lk - 1, Lk - 1);
        }
      }
      release_item(sm, taken, lane);
      ++taken;
      if (id < 0) break;
      const bool row_valid = row >= 0;
      uint4 *dst = reinterpret_cast<uint4 *>(p.out + (row_valid ? row : 0) * kD);
      if (nk == 0) {  // no key is visible to any row: zeros
        if (row_valid)
          for (int c = 0; c < 16; ++c) dst[c] = make_uint4(0, 0, 0, 0);
        continue;
      }
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < nk; ++j, ++g) {
        // warp-uniform results: the TMEM loads and stores below are .sync.aligned
        ok = __all_sync(kFull, wait_parity(&sm.s_full[a], g & 1, p.err));
        if (!ok) break;
        tc_fence_after_sync();
        const int64_t rel = lim - (int64_t)j * kBN;  // last visible column of this tile
        const int lim_rel = (int)(rel < -1 ? -1 : (rel > kBN ? kBN : rel));

        // the whole S row in registers: one TMEM round trip per tile
        uint32_t x[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(lane_addr + s_col + 32 * c, x[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_wait(x[c]);
        if (lim_rel < kBN - 1) {  // diagonal or last tile: columns past lim_rel are -inf
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (32 * c + e > lim_rel) x[c][e] = __float_as_uint(-INFINITY);
        }
        float mx[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          mx[c] = -INFINITY;
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            mx[c] = fmax3(mx[c], __uint_as_float(x[c][e]), __uint_as_float(x[c][e + 1]));
        }
        const float m_tile = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3])) * p.scale_log2;
        const float m_new = fmaxf(m_run, m_tile);
        const bool rescale = m_new > m_run + kRescaleLog2;
        float alpha = 1.f;
        if (rescale) {
          alpha = fast_exp2(m_run - m_new);
          m_run = m_new;
          l_run *= alpha;
        }
        const float neg_m = m_run == -INFINITY ? 0.f : -m_run;

        // O_a holds the tiles before this one: rescale it (never on the first tile)
        if (j > 0 && __any_sync(kFull, rescale)) {
          ok = __all_sync(kFull, wait_parity(&sm.o_full[a], (g - 1) & 1, p.err));
          if (!ok) break;
          tc_fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(lane_addr + o_col + 32 * c, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(lane_addr + o_col + 32 * c, o);
          }
        }

        // P = 2^(s * scale_log2 - m) as bf16 pairs over the first 64 columns of S
        const float2 nm2 = make_float2(neg_m, neg_m);
        float2 rs0 = make_float2(0.f, 0.f), rs1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 t = ffma2(make_float2(__uint_as_float(x[c][2 * e]),
                                               __uint_as_float(x[c][2 * e + 1])), sl2, nm2);
            const float2 pe = make_float2(fast_exp2(t.x), fast_exp2(t.y));
            if (e & 1) rs1 = fadd2(rs1, pe);
            else rs0 = fadd2(rs0, pe);
            pk[e] = pack_bf16(pe.x, pe.y);
          }
          tmem_st16(lane_addr + s_col + 16 * c, pk);
        }
        tmem_st_wait();
        l_run += (rs0.x + rs0.y) + (rs1.x + rs1.y);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_full[a]);
      }
      if (!ok) break;
      // ---- epilogue: O / l -> bf16 rows
      ok = __all_sync(kFull, wait_parity(&sm.o_full[a], (g - 1) & 1, p.err));
      if (!ok) break;
      tc_fence_after_sync();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(lane_addr + o_col + 32 * c, o);
        tmem_ld_wait(o);
        if (row_valid) {
          // a thread writes its own row: one 32-byte sector per store when out allows it
          // (a warp's store touches 32 rows, so fewer and wider stores leave the load/store
          // queue free sooner for the TMEM, shared-memory and UMMA traffic behind them)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              w[k] = pack_bf16(__uint_as_float(o[16 * e + 2 * k]) * inv,
                               __uint_as_float(o[16 * e + 2 * k + 1]) * inv);
            uint4 *d = dst + c * 4 + 2 * e;
            if (p.out_32b) {
              st_global_32b(d, w);
            } else {
              d[0] = make_uint4(w[0], w[1], w[2], w[3]);
              d[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
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

// ---------------------------------------------------------------------- work-list planner
struct PlanParams {
  const int32_t *cu_q;
  int32_t num_seqs;
  int32_t levels;           // most query blocks a sequence may have
  int32_t tokens_per_unit;  // query rows of one unit (128, or 256 without GQA pairs)
  int64_t total_q;
  int32_t *header;          // [0] work counter, [1] number of units
  int32_t *counts, *ranked, *unit_start, *hist, *fill;
  int2 *units;
  unsigned int *err;
};
constexpr int kPlanThreads = 1024;

// Exclusive prefix sum of one value per thread over the block; `total` gets the block's sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_sums, int &total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  const int base = warp > 0 ? warp_sums[warp - 1] : 0;
  total = warp_sums[31];
  __syncthreads();  // warp_sums is reused by the next call
  return base + x - v;
}

// One CTA: count each sequence's query blocks, rank the sequences by that count (most first;
// a counting sort), and write the unit list. Sequences whose cu_seqlens_q are inconsistent
// get no units and set PKV_DEVERR_SEQLEN_RANGE, as does a sequence longer than the host's
// max_seqlen_q (its blocks past that bound are dropped).
__global__ void __launch_bounds__(kPlanThreads, 1) prefill_plan_kernel(const PlanParams p) {
  __shared__ int warp_sums[32];
  const int tid = threadIdx.x;
  for (int c = tid; c <= p.levels; c += kPlanThreads) {
    p.hist[c] = 0;
    p.fill[c] = 0;
  }
  __syncthreads();
  for (int n = tid; n < p.num_seqs; n += kPlanThreads) {
    const int64_t a = p.cu_q[n], b = p.cu_q[n + 1];
    int c = 0;
    if (a < 0 || b < a || b > p.total_q) {
      record_error(p.err, 8u /* SEQLEN_RANGE */);
    } else {
      const int64_t cc = (b - a + p.tokens_per_unit - 1) / p.tokens_per_unit;
      if (cc > p.levels) record_error(p.err, 8u /* SEQLEN_RANGE */);
      c = (int)min(cc, (int64_t)p.levels);
    }
    p.counts[n] = c;
    atomicAdd(&p.hist[c], 1);
  }
  __syncthreads();
  // first rank of each count: the sequences with a larger count come before it
  int carry = 0;
  for (int r0 = 0; r0 <= p.levels; r0 += kPlanThreads) {
    const int r = r0 + tid, c = p.levels - r;
    int total;
    const int ex = block_exclusive_scan(r <= p.levels ? p.hist[c] : 0, warp_sums, total);
    if (r <= p.levels) p.fill[c] = carry + ex;
    carry += total;
  }
  __syncthreads();
  for (int n = tid; n < p.num_seqs; n += kPlanThreads)
    p.ranked[atomicAdd(&p.fill[p.counts[n]], 1)] = n;
  __syncthreads();
  // first unit of each ranked sequence
  carry = 0;
  for (int k0 = 0; k0 < p.num_seqs; k0 += kPlanThreads) {
    const int k = k0 + tid;
    int total;
    const int ex = block_exclusive_scan(k < p.num_seqs ? p.counts[p.ranked[k]] : 0, warp_sums,
                                        total);
    if (k < p.num_seqs) p.unit_start[k] = carry + ex;
    carry += total;
  }
  __syncthreads();
  // the units of each ranked sequence, its last query block first
  const int warp = tid >> 5, lane = tid & 31;
  for (int k = warp; k < p.num_seqs; k += kPlanThreads / 32) {
    const int n = p.ranked[k], c = p.counts[n], base = p.unit_start[k];
    for (int u = lane; u < c; u += 32) p.units[base + u] = make_int2(n, c - 1 - u);
  }
  if (tid == 0) {
    p.unit_start[p.num_seqs] = carry;
    p.header[0] = 0;
    p.header[1] = carry;
  }
}

template <int G>
cudaError_t launch_g(const PrefillArgs &a, PrefillParams prm, int num_sms, cudaStream_t stream) {
  constexpr int kPairs = G >= 2 ? G / 2 : 1;
  constexpr int kTokensPerItem = G >= 2 ? kBM : 2 * kBM;
  CUtensorMap qm, km, vm;
  const uint64_t qdims[3] = {64, (uint64_t)a.total_q, (uint64_t)a.num_q_heads * 2};
  const uint64_t qstr[2] = {(uint64_t)a.q_tok_stride * 2, 128};
  const uint32_t qbox[3] = {64, (uint32_t)kBM, 1};
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
    // The register split inside the kernel draws on the registers the CTA is launched with;
    // never launch a build whose count cannot cover it (the increase would never return).
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, prefill_kernel<G>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * kThreads < (2 * kSoftmaxRegs + kOtherRegs) * 128)
      return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(prefill_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const PrefillWorkspace wl = prefill_workspace_layout(a.num_seqs, a.max_seqlen_q);
  uint8_t *ws = static_cast<uint8_t *>(a.workspace);
  PlanParams pp{};
  pp.cu_q = a.cu_seqlens_q;
  pp.num_seqs = a.num_seqs;
  pp.levels = wl.levels;
  pp.tokens_per_unit = kTokensPerItem;
  pp.total_q = a.total_q;
  pp.header = reinterpret_cast<int32_t *>(ws);
  pp.counts = reinterpret_cast<int32_t *>(ws + wl.counts);
  pp.ranked = reinterpret_cast<int32_t *>(ws + wl.ranked);
  pp.unit_start = reinterpret_cast<int32_t *>(ws + wl.unit_start);
  pp.hist = reinterpret_cast<int32_t *>(ws + wl.hist);
  pp.fill = reinterpret_cast<int32_t *>(ws + wl.fill);
  pp.units = reinterpret_cast<int2 *>(ws + wl.units);
  pp.err = a.err;
  prm.queue = pp.header;
  prm.num_units = pp.header + 1;
  prm.units = pp.units;
  const int64_t items = wl.max_units * a.num_kv_heads * kPairs;  // an upper bound
  if (items <= 0) return cudaSuccess;
  if (items > INT32_MAX) return cudaErrorInvalidValue;
  const unsigned grid = (unsigned)(items < num_sms ? items : num_sms);
  prefill_plan_kernel<<<1, kPlanThreads, 0, stream>>>(pp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prefill_kernel<G><<<grid, kThreads, smem, stream>>>(qm, km, vm, prm);
  return cudaGetLastError();
}

}  // namespace

bool prefill_group_supported(int group) {
  return group == 1 || group == 2 || group == 4 || group == 8;
}

cudaError_t launch_varlen_prefill(const PrefillArgs &a, int num_sms, cudaStream_t stream) {
  PrefillParams prm{};
  prm.cu_q = a.cu_seqlens_q;
  prm.cu_k = a.cu_seqlens_k;
  prm.block_table = a.block_table;
  prm.table_width = a.table_width;
  prm.block_size = a.block_size;
  prm.num_blocks = a.num_blocks;
  prm.total_q = a.total_q;
  prm.kv_rows = a.kv_rows;
  prm.num_seqs = a.num_seqs;
  prm.num_q_heads = a.num_q_heads;
  prm.num_kv_heads = a.num_kv_heads;
  prm.scale_log2 = a.scale * kLog2e;
  prm.causal = a.causal;
  prm.out = static_cast<uint16_t *>(a.out);
  prm.out_32b = (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0;
  prm.err = a.err;
  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_g<1>(a, prm, num_sms, stream);
    case 2: return launch_g<2>(a, prm, num_sms, stream);
    case 4: return launch_g<4>(a, prm, num_sms, stream);
    case 8: return launch_g<8>(a, prm, num_sms, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace pkv
