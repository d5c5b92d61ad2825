// prefill.cu -- varlen causal prefill attention on the 5th-generation tensor cores (sm_103a).
//
// flash_attn_varlen_func of «nano-vLLM 最小化vLLM重新实现», 架构 5: causal attention over
// cu_seqlens-packed prompts, keys either packed or read from the paged pool through a block
// table (prefix caching: queries cover only the uncached suffix and the causal mask is
// aligned to the end of the keys).
//
// Persistent kernel on CTA pairs (clusters of two CTAs, each on its own SM). A one-CTA
// planning kernel first writes the work list into the caller's workspace: only (sequence,
// query block) units that have queries, sequences with the most query blocks first and each
// sequence's blocks heaviest first, all heads of a unit next to each other, so the heavy work
// starts first and the query blocks of one sequence run at about the same time (their K/V
// tiles come from L2). The pair's leader takes items from a global counter and hands them to
// both CTAs. An item is one sequence n, one KV head h and 256 query rows: for a GQA group of
// two (or a pair of heads of a larger group) the two query heads over the same 128 tokens,
// without GQA two consecutive 128-token blocks of the one head; the leader holds the first
// 128 rows, the peer the other 128. Per 128-key tile j, with M = 256 over the pair:
//   S(j) = Q K_j^T     tcgen05.mma.cta_group::2: each CTA's 128 Q rows from its own shared
//                      memory, K_j split by key (leader keys 0-63, peer 64-127), S rows into
//                      each CTA's tensor memory
//   softmax            one warpgroup per CTA, thread = row: row max and P = 2^(s - m) read
//                      from TMEM with tcgen05.ld, P written back as bf16 over S's first 64
//                      columns
//   O += P V_j         A = P from each CTA's tensor memory, V_j split by head dimension
//                      (leader dims 0-63, peer 64-127)
// S has three buffers in tensor memory, so the tensor core computes S(j+1) and S(j+2) while
// the softmax works on S(j): S(j+3), which reuses P(j)'s buffer, is issued once PV(j) has
// completed, across item boundaries. O is rescaled in TMEM only when a row's running max grows
// by more than 2^8 (its sum l carries the same stale max, so O / l is unchanged). At an item
// switch the softmax warps first compute the next item's first P, then read the finished O,
// release it (the next item's first PV waits for that) and write it out, so the tensor core
// has work queued while the epilogue runs.
//
// Warps (384 threads per CTA): 0-7 softmax and epilogue (warp w: 16 rows of TMEM lane
// quadrant w % 4, two threads per row), 8 Q and K loads (Q per item, this CTA's K half per key
// tile through a 5-slot ring; in the leader also the scheduler), 10 V loads (this CTA's V half
// per key tile through a 4-slot ring, which lets V tiles, needed three tiles after their K, be
// loaded later), 9 and 11 in the leader the S and the PV issuers; in the peer warp 9 is a
// relay that forwards the peer's load completions to the leader's load barriers. All loads are
// TMA with 128-byte swizzle. Every load lands on a barrier of the CTA that issued it, so each
// CTA can wait for its own copies before it exits, whatever the other one does.
// TMEM (512 columns per CTA): S buffers [0,128), [128,256), [256,384), O [384,512). Shared
// memory per CTA: two Q buffers of 32 KiB, five K and four V slots of 16 KiB.
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
constexpr int kBM = 128;   // query rows per CTA (M = 256 per pair)
constexpr int kBN = 128;   // keys per tile
constexpr int kKSlots = 5;  // K ring: K(t) in slot t % 5 (needed by S(t))
constexpr int kVSlots = 4;  // V ring: V(t) in slot t % 4 (needed by PV(t), three tiles later)
constexpr int kSBufs = 3;   // S buffers in tensor memory
constexpr int kSoftmaxWarps = 8;
constexpr int kKLoadWarp = 8;
constexpr int kSMmaWarp = 9;   // the relay in the peer
constexpr int kVLoadWarp = 10;
constexpr int kPvMmaWarp = 11;  // idle in the peer
constexpr int kThreads = 12 * 32;
constexpr uint32_t kQBytes = kBM * kD * 2;     // 32 KiB: one CTA's Q rows
constexpr uint32_t kQHalf = kQBytes / 2;       // one 64-dim half of them
constexpr uint32_t kSlotBytes = 16384;         // one CTA's half of a K or V tile
constexpr uint32_t kKHalf = kSlotBytes / 2;    // one 64-dim half of a K half-tile (64 keys)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 384;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kRing = 8;   // work items in flight between the scheduler and the other warps
// item_empty arrivals: leader S and PV issuers, V loader and 8 softmax warps; peer K loader,
// V loader, relay and 8 softmax warps
constexpr int kItemConsumers = 22;
constexpr int kSoftmaxArrivals = 2 * kSoftmaxWarps;  // per P / per O release, both CTAs

// A work item as the scheduler hands it out (16 words, copied to both CTAs of the pair).
struct Item {
  int32_t id;         // index in the work list; -1 marks the end of the work
  int32_t n, h;
  int32_t hq[2];      // query head of the leader's and of the peer's rows
  int32_t tok[2];     // first query token (within the sequence) of each CTA's rows
  int32_t q0, Lq, k0, Lk;
  int32_t nk;         // key tiles to process
  int32_t last_rows;  // keys of the sequence in the last key tile
  int32_t valid;      // the item has queries
  int32_t bad;        // cu_seqlens / block_table inconsistent for this sequence
  int32_t pad;
};
static_assert(sizeof(Item) == 64, "Item is copied to the peer as four 16-byte words");

struct PrefillSmem {
  uint8_t q[2][kQBytes];            // 1024-byte aligned (128-byte swizzle atoms)
  uint8_t k[kKSlots][kSlotBytes];
  uint8_t v[kVSlots][kSlotBytes];
  alignas(16) Item items[kRing];    // written by the leader's scheduler into both CTAs
  // this CTA's loads; in the leader each phase also waits for the relay's arrival, which
  // says that the peer's half of the same load has landed (two arrivals per phase)
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kKSlots], k_empty[kKSlots], v_full[kVSlots], v_empty[kVSlots];
  // leader only: the V fixes of both CTAs, the softmax warps' P of each S buffer and their
  // release of O, the MMA drain
  uint64_t v_fixed[kVSlots];
  uint64_t p_full[kSBufs], o_free, mma_drain[2];
  // both CTAs, committed by the leader's MMA thread: S(t) and PV(t) done, per S buffer t % 3
  // (a parity wait only tells the current phase from the one before, and the softmax warps
  // can be two tiles ahead of the last finished PV)
  uint64_t s_full[kSBufs], o_full[kSBufs];
  uint64_t item_full[kRing], item_empty[kRing];
  uint32_t tmem_base;
  int32_t stop;                     // the cluster returns at once (an earlier wait gave up)
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
  int32_t *queue;  // next item to hand out (zeroed by the planner)
  unsigned int *err;
};

// Item i of the work list: unit i / (KV heads x head pairs), head pair i % that.
template <int G>
__device__ __forceinline__ Item decode_item(const PrefillParams &p, int i) {
  constexpr int kPairs = G >= 2 ? G / 2 : 1;
  Item it;
  it.id = i;
  it.pad = 0;
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
    it.tok[0] = it.tok[1] = qb * kBM;
  } else {
    it.hq[0] = it.hq[1] = it.h;
    it.tok[0] = qb * 2 * kBM;
    it.tok[1] = it.tok[0] + kBM;
  }
  const int64_t q0 = p.cu_q[it.n], Lq = p.cu_q[it.n + 1] - q0;
  const int64_t k0 = p.cu_k[it.n], Lk = p.cu_k[it.n + 1] - k0;
  bool bad = Lq < 0 || Lk < 0 || q0 < 0 || q0 + Lq > p.total_q;
  if (p.block_table) bad = bad || Lk > (int64_t)p.table_width * p.block_size;
  else bad = bad || k0 < 0 || k0 + Lk > p.kv_rows;
  it.q0 = (int32_t)q0;
  it.Lq = (int32_t)Lq;
  it.k0 = (int32_t)k0;
  it.Lk = (int32_t)Lk;
  it.bad = bad;
  it.valid = !bad && it.tok[0] < Lq;
  it.nk = 0;
  it.last_rows = 0;
  if (it.valid) {
    int64_t kv_end = 0;
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      if (it.tok[a] >= Lq) continue;
      const int64_t last_q = min(Lq, (int64_t)it.tok[a] + kBM) - 1;
      const int64_t e = p.causal ? min(Lk, last_q + (Lk - Lq) + 1) : Lk;
      kv_end = max(kv_end, e);
    }
    if (kv_end > 0) {
      it.nk = (int)((kv_end + kBN - 1) / kBN);
      it.last_rows = (int)min((int64_t)kBN, Lk - (int64_t)(it.nk - 1) * kBN);
    }
  }
  return it;
}

// Next work item from this CTA's ring (in order), taken by a whole warp: every lane waits,
// and the item counts only if every lane saw it. In the peer the leader's scheduler wrote
// the item with remote stores, so the wait acquires at cluster scope there. Returns the
// slot, or nullptr when the wait gave up.
__device__ __forceinline__ const Item *wait_item(PrefillSmem &sm, uint32_t taken, bool leader,
                                                 unsigned int *err) {
  const int slot = taken % kRing;
  const uint32_t par = (taken / kRing) & 1;
  if (__all_sync(kFull, leader ? wait_parity(&sm.item_full[slot], par, err)
                               : wait_parity_cluster(&sm.item_full[slot], par, err)))
    return &sm.items[slot];
  return nullptr;
}

// Release a ring slot once every lane has read it: one arrival per warp on the leader's
// item_empty (item_empty_l = its shared::cluster address).
__device__ __forceinline__ void release_item(uint32_t item_empty_l, uint32_t taken, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive_remote(item_empty_l + (taken % kRing) * 8);
}

// S = Q K^T for one tile over the pair: 8 UMMAs of K = 16 over the two 64-dim halves. The
// descriptors are the tiles' base descriptors plus compile-time offsets (the start address
// sits in the low bits, in 16-byte units). Issued by the MMA warp's elected lane.
__device__ __forceinline__ void mma_qk(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc,
                                       uint32_t idesc) {
  umma_pair_ss<false>(d_tmem, q_desc, k_desc, idesc);
#pragma unroll
  for (int kk = 1; kk < kD / 16; ++kk) {
    const uint64_t qoff = ((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4;
    const uint64_t koff = ((kk >> 2) * kKHalf + (kk & 3) * 32) >> 4;
    umma_pair_ss<true>(d_tmem, q_desc + qoff, k_desc + koff, idesc);
  }
}

// O (+)= P V for one tile: P from TMEM (8 columns per 16 keys), V MN-major in shared memory
// (16 keys = 2 KiB further per step).
__device__ __forceinline__ void mma_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t v_desc,
                                       uint32_t idesc, bool accumulate) {
  if (accumulate) umma_pair_ts<true>(d_tmem, p_tmem, v_desc, idesc);
  else umma_pair_ts<false>(d_tmem, p_tmem, v_desc, idesc);
#pragma unroll
  for (int kk = 1; kk < kBN / 16; ++kk)
    umma_pair_ts<true>(d_tmem, p_tmem + 8 * kk, v_desc + ((kk * 16 * 128) >> 4), idesc);
}

// Commits to the barrier at the same offset in both CTAs (bar_l = its address in the leader,
// bar_p in the peer).
__device__ __forceinline__ void commit_both(uint32_t bar_l, uint32_t bar_p) {
  umma_commit_pair(bar_l);
  umma_commit_pair(bar_p);
}

// Time limit of the loaders' final waits for their own loads. In the leader a load's phase
// also needs the relay's arrival for the peer's half; after an abort that arrival may never
// come, while the leader's own bytes land within microseconds of being issued, so there the
// wait is cut to 1 ms.
__device__ __forceinline__ uint64_t drain_limit_ns(const unsigned int *err, bool leader) {
  return leader && aborted(err) ? 1000000ull : kWaitLimitNs;
}

// First pool (or packed) row of key tile j of an item; a block id outside the pool is
// flagged and gives a row wholly outside the tensor (TMA fills zeros there).
__device__ __forceinline__ int32_t tile_row(const PrefillParams &p, const Item &it, int j) {
  if (!p.block_table) return it.k0 + j * kBN;
  const int64_t key = (int64_t)j * kBN;
  const int64_t blk = p.block_table[(int64_t)it.n * p.table_width + key / p.block_size];
  if (blk < 0 || blk >= p.num_blocks) {
    record_error(p.err, 2u /* BLOCK_RANGE */);
    return -2 * kBN;
  }
  return (int32_t)(blk * p.block_size + key % p.block_size);
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
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  extern __shared__ uint8_t smem_raw[];
  PrefillSmem &sm = *reinterpret_cast<PrefillSmem *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  if (tid == 0) {
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sm.q_full[a], leader ? 2 : 1);
      mbar_init(&sm.q_empty[a], 1);
    }
    for (int i = 0; i < kKSlots; ++i) {
      mbar_init(&sm.k_full[i], leader ? 2 : 1);
      mbar_init(&sm.k_empty[i], 1);
    }
    for (int i = 0; i < kVSlots; ++i) {
      mbar_init(&sm.v_full[i], leader ? 2 : 1);
      mbar_init(&sm.v_empty[i], 1);
      mbar_init(&sm.v_fixed[i], 2);
    }
    for (int b = 0; b < kSBufs; ++b) {
      mbar_init(&sm.s_full[b], 1);
      mbar_init(&sm.p_full[b], kSoftmaxArrivals);
      mbar_init(&sm.o_full[b], 1);
    }
    mbar_init(&sm.o_free, kSoftmaxArrivals);
    mbar_init(&sm.mma_drain[0], 1);
    mbar_init(&sm.mma_drain[1], 1);
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&sm.item_full[i], 1);
      mbar_init(&sm.item_empty[i], kItemConsumers);
    }
    fence_mbar_init();
  }
  // Both CTAs have started and initialised their barriers; then the leader decides for the
  // pair whether an earlier wait gave up (the whole cluster returns before allocating).
  cluster_sync();
  if (leader && tid == 0) {
    const int32_t stop = aborted(p.err) ? 1 : 0;
    sm.stop = stop;
    st_cluster_u32(cluster_addr(smem_addr(&sm.stop), 1), (uint32_t)stop);
  }
  cluster_sync();
  if (sm.stop) return;
  if (warp == kSMmaWarp) {
    tmem_alloc_pair(&sm.tmem_base, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t item_empty_l = cluster_addr(smem_addr(&sm.item_empty[0]), 0);
  const uint32_t p_full_l = cluster_addr(smem_addr(&sm.p_full[0]), 0);
  const uint32_t o_free_l = cluster_addr(smem_addr(&sm.o_free), 0);
  constexpr int kPairs = G >= 2 ? G / 2 : 1;

  if (warp == kKLoadWarp) {
    // ---------------------------------------- scheduler (leader) + Q and K loads (both CTAs)
    // Lane 0 takes the items (in the leader) and issues the loads; the whole warp runs the
    // loop so that every lane sees the same decisions.
    uint64_t pol_q = 0, pol_kv = 0;
    if (lane == 0) {
      prefetch_tensormap(&qmap);
      prefetch_tensormap(&kmap);
      pol_q = policy_evict_first();
      pol_kv = policy_evict_last();
    }
    uint32_t taken = 0, q_loads = 0, g = 0;
    uint32_t q_issued[2] = {0, 0};  // loads issued into each Q buffer (lane 0's count)
    uint32_t k_issued = 0;          // K loads issued (in tile order)
    bool ok = true;
    const int total_items =
        (leader && lane == 0) ? *p.num_units * p.num_kv_heads * kPairs : 0;
    while (ok) {
      const int slot = taken % kRing;
      if (leader) {
        // take the next item that has queries; id -1 when the queue is exhausted
        if (lane == 0) {
          Item d;
          int i;
          while (true) {
            i = atomicAdd(p.queue, 1);
            if (i >= total_items) break;
            d = decode_item<G>(p, i);
            if (d.bad) record_error(p.err, 8u /* SEQLEN_RANGE */);
            if (d.valid) break;
          }
          if (i >= total_items) {
            d = Item{};
            d.id = -1;
          }
          if (taken >= kRing)
            ok = wait_parity_cluster(&sm.item_empty[slot], ((taken / kRing) - 1) & 1, p.err);
          if (ok) {
            sm.items[slot] = d;
            const uint32_t dst = cluster_addr(smem_addr(&sm.items[slot]), 1);
            const uint4 *w4 = reinterpret_cast<const uint4 *>(&d);
#pragma unroll
            for (int k = 0; k < 4; ++k) st_cluster_v4(dst + 16 * k, w4[k]);
            mbar_arrive(&sm.item_full[slot]);  // release: visible to this CTA's waiters
            mbar_arrive_cluster(cluster_addr(smem_addr(&sm.item_full[slot]), 1));
          }
        }
        ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        __syncwarp();  // lane 0 wrote the slot
      } else {
        ok = __all_sync(kFull, wait_parity_cluster(&sm.item_full[slot], (taken / kRing) & 1, p.err));
        if (!ok) break;
      }
      const Item it = sm.items[slot];
      if (!leader) release_item(item_empty_l, taken, lane);
      ++taken;
      if (it.id < 0) break;
      if (it.nk == 0) continue;  // no key visible: the softmax warps write zeros
      if (lane == 0) {
        const int qb = q_loads & 1;
        if (q_loads >= 2) ok = wait_parity(&sm.q_empty[qb], ((q_loads >> 1) - 1) & 1, p.err);
        if (ok) {
          mbar_arrive_expect_tx(&sm.q_full[qb], kQBytes);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
            tma_load_3d(sm.q[qb] + hf * kQHalf, &qmap, &sm.q_full[qb], 0,
                        it.q0 + it.tok[rank], 2 * it.hq[rank] + hf, pol_q);
          ++q_issued[qb];
        }
        for (int j = 0; j < it.nk && ok; ++j, ++g) {
          const int ks = g % kKSlots;
          if (g >= kKSlots) ok = wait_parity(&sm.k_empty[ks], ((g / kKSlots) - 1) & 1, p.err);
          if (ok) {  // this CTA's 64 keys: both 64-dim halves in one box
            mbar_arrive_expect_tx(&sm.k_full[ks], kSlotBytes);
            tma_load_3d(sm.k[ks], &kmap, &sm.k_full[ks], 0,
                        tile_row(p, it, j) + 64 * (int32_t)rank, 2 * it.h, pol_kv);
            ++k_issued;
          }
        }
      }
      ++q_loads;
      ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
      g = __shfl_sync(kFull, g, 0);
    }
    if (lane == 0) {
      // keep the CTA alive until every copy it issued has landed, also after an abort (these
      // waits ignore the abort bit; only issued loads are waited for)
      const uint64_t lim = drain_limit_ns(p.err, leader);
      bool drained = true;
      for (int a = 0; a < 2; ++a)
        if (q_issued[a] > 0)
          drained = drained && wait_own(&sm.q_full[a], (q_issued[a] - 1) & 1, p.err, lim);
      for (uint32_t t = k_issued > kKSlots ? k_issued - kKSlots : 0; drained && t < k_issued; ++t)
        drained = wait_own(&sm.k_full[t % kKSlots], (t / kKSlots) & 1, p.err, lim);
    }
    __syncwarp();
  } else if (warp == kVLoadWarp) {
    // ---------------------------------------------------------------- V loads (both CTAs)
    // Follows the items on its own ring, so V tiles (needed three tiles after their K) are
    // loaded as late as the V ring allows; zeroes the rows of an item's last V tile past
    // the sequence's keys (the whole warp), then tells the leader's MMA thread.
    uint64_t pol_kv = 0;
    if (lane == 0) {
      prefetch_tensormap(&vmap);
      pol_kv = policy_evict_last();
    }
    const uint32_t v_fixed_l = cluster_addr(smem_addr(&sm.v_fixed[0]), 0);
    uint32_t taken = 0, g = 0, v_issued = 0;
    bool ok = true;
    while (ok) {
      const Item *ip = wait_item(sm, taken, leader, p.err);
      if (!ip) break;
      const Item it = *ip;
      release_item(item_empty_l, taken, lane);
      ++taken;
      if (it.id < 0) break;
      for (int j = 0; j < it.nk && ok; ++j, ++g) {
        const int vs = g % kVSlots;
        if (lane == 0) {
          if (g >= kVSlots) ok = wait_parity(&sm.v_empty[vs], ((g / kVSlots) - 1) & 1, p.err);
          if (ok) {  // this CTA's 64 dims of all 128 keys
            mbar_arrive_expect_tx(&sm.v_full[vs], kSlotBytes);
            tma_load_3d(sm.v[vs], &vmap, &sm.v_full[vs], 0, tile_row(p, it, j),
                        2 * it.h + (int32_t)rank, pol_kv);
            ++v_issued;
          }
        }
        ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
        if (ok && j == it.nk - 1 && it.last_rows < kBN) {
          ok = __all_sync(kFull, wait_parity(&sm.v_full[vs], (g / kVSlots) & 1, p.err));
          if (ok) {
            uint8_t *vt = sm.v[vs];
            for (int idx = lane; idx < (kBN - it.last_rows) * 8; idx += 32)
              *reinterpret_cast<uint4 *>(vt + (it.last_rows + (idx >> 3)) * 128 + (idx & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
            fence_async_shared();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(v_fixed_l + vs * 8);
          }
        }
      }
    }
    if (lane == 0) {  // drain this CTA's V loads (ignores the abort bit)
      const uint64_t lim = drain_limit_ns(p.err, leader);
      bool drained = true;
      for (uint32_t t = v_issued > kVSlots ? v_issued - kVSlots : 0; drained && t < v_issued; ++t)
        drained = wait_own(&sm.v_full[t % kVSlots], (t / kVSlots) & 1, p.err, lim);
    }
    __syncwarp();
  } else if (warp == kSMmaWarp && !leader) {
    // ------------------------------------------------------------------ relay (peer)
    // Forward each of this CTA's Q, K and V loads to the leader once it has landed. One lane
    // polls the three streams (each in load order) without blocking, so a load that lands
    // early is never held up behind another stream's; it learns the loads from the item
    // ring and sleeps briefly when nothing is ready. Gives up like a wait: after the time
    // limit without progress, or at once when the abort bit is set.
    if (lane == 0) {
      const uint32_t q_full_l = cluster_addr(smem_addr(&sm.q_full[0]), 0);
      const uint32_t k_full_l = cluster_addr(smem_addr(&sm.k_full[0]), 0);
      const uint32_t v_full_l = cluster_addr(smem_addr(&sm.v_full[0]), 0);
      uint32_t taken = 0, q_known = 0, t_known = 0, q_next = 0, k_next = 0, v_next = 0;
      bool end = false;
      uint64_t t0 = global_timer_ns();
      while (true) {
        bool progressed = false;
        if (!end && mbar_test_wait(&sm.item_full[taken % kRing], (taken / kRing) & 1) &&
            mbar_test_wait_cluster(&sm.item_full[taken % kRing], (taken / kRing) & 1)) {
          const Item &it = sm.items[taken % kRing];
          const int id = it.id, nk = it.nk;
          mbar_arrive_remote(item_empty_l + (taken % kRing) * 8);
          ++taken;
          if (id < 0) {
            end = true;
          } else if (nk > 0) {
            ++q_known;
            t_known += nk;
          }
          progressed = true;
        }
        if (q_next < q_known && mbar_test_wait(&sm.q_full[q_next & 1], (q_next >> 1) & 1)) {
          mbar_arrive_remote(q_full_l + (q_next & 1) * 8);
          ++q_next;
          progressed = true;
        }
        if (k_next < t_known &&
            mbar_test_wait(&sm.k_full[k_next % kKSlots], (k_next / kKSlots) & 1)) {
          mbar_arrive_remote(k_full_l + (k_next % kKSlots) * 8);
          ++k_next;
          progressed = true;
        }
        if (v_next < t_known &&
            mbar_test_wait(&sm.v_full[v_next % kVSlots], (v_next / kVSlots) & 1)) {
          mbar_arrive_remote(v_full_l + (v_next % kVSlots) * 8);
          ++v_next;
          progressed = true;
        }
        if (end && q_next == q_known && k_next == t_known && v_next == t_known) break;
        if (progressed) {
          t0 = global_timer_ns();
        } else {
          if (aborted(p.err)) break;
          if (global_timer_ns() - t0 > kWaitLimitNs) {
            record_error(p.err, kErrTimeout);
            break;
          }
          __nanosleep(32);
        }
      }
    }
    __syncwarp();
  } else if (leader && (warp == kSMmaWarp || warp == kPvMmaWarp)) {
    // ------------------------------------------------------------- UMMA issuers (leader)
    // Two warps on different SM sub-partitions: one issues S = Q K^T for every tile, the other
    // O += P V. S(t) reuses the tensor-memory buffer of P(t - 3), so the S warp waits for
    // PV(t - 3) to complete first. Each warp runs its loop converged and one elected lane
    // issues a step's UMMAs and commits (commits track the issuing thread's UMMAs; the warp
    // is converged at every elect, so it is always the same lane).
    const bool s_role = warp == kSMmaWarp;
    uint64_t *drain_bar = s_role ? &sm.mma_drain[0] : &sm.mma_drain[1];
    auto wait_all = [&](uint64_t *bar, uint32_t parity) -> bool {
      return __all_sync(kFull, wait_parity(bar, parity, p.err));
    };
    const uint32_t o_full_l = cluster_addr(smem_addr(&sm.o_full[0]), 0);
    const uint32_t o_full_p = cluster_addr(smem_addr(&sm.o_full[0]), 1);
    uint32_t taken = 0;
    bool ok = true;
    if (s_role) {
      constexpr uint32_t kIdS = idesc_bf16_f32(2 * kBM, kBN, 0, 0);  // Q (K-major) x K (K-major)
      const uint64_t dq0 = smem_desc_sw128(smem_addr(sm.q[0]), 16, 1024);
      const uint64_t dq1 = smem_desc_sw128(smem_addr(sm.q[1]), 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(smem_addr(sm.k[0]), 16, 1024);
      const uint32_t s_full_l = cluster_addr(smem_addr(&sm.s_full[0]), 0);
      const uint32_t s_full_p = cluster_addr(smem_addr(&sm.s_full[0]), 1);
      const uint32_t k_empty_l = cluster_addr(smem_addr(&sm.k_empty[0]), 0);
      const uint32_t k_empty_p = cluster_addr(smem_addr(&sm.k_empty[0]), 1);
      const uint32_t q_empty_l = cluster_addr(smem_addr(&sm.q_empty[0]), 0);
      const uint32_t q_empty_p = cluster_addr(smem_addr(&sm.q_empty[0]), 1);
      uint32_t t = 0, items_nz = 0, q_use0 = 0, q_use1 = 0;
      while (ok) {
        const Item *ip = wait_item(sm, taken, leader, p.err);
        const int id = ip ? ip->id : -1, nk = ip ? ip->nk : 0;
        release_item(item_empty_l, taken, lane);
        ++taken;
        if (!ip) {
          ok = false;
          break;
        }
        if (id < 0) break;
        if (nk == 0) continue;
        const int qb = items_nz & 1;
        ++items_nz;
        const uint32_t q_use = qb ? q_use1 : q_use0;
        for (int j = 0; j < nk && ok; ++j, ++t) {
          const uint32_t ks = t % kKSlots, sb = t % kSBufs;
          ok = wait_all(&sm.k_full[ks], (t / kKSlots) & 1);
          if (ok && j == 0) ok = wait_all(&sm.q_full[qb], q_use & 1);
          // the buffer's previous P has been read by its PV
          if (ok && t >= kSBufs) ok = wait_all(&sm.o_full[sb], ((t - kSBufs) / kSBufs) & 1);
          if (!ok) break;
          tc_fence_after_sync();
          const bool last = j == nk - 1;
          if (elect_one()) {
            mma_qk(tmem + 128 * sb, qb ? dq1 : dq0, dk0 + ks * (kSlotBytes >> 4), kIdS);
            commit_both(s_full_l + 8 * sb, s_full_p + 8 * sb);
            commit_both(k_empty_l + 8 * ks, k_empty_p + 8 * ks);
            if (last) commit_both(q_empty_l + 8 * qb, q_empty_p + 8 * qb);
          }
          __syncwarp();
        }
        if (qb) ++q_use1;
        else ++q_use0;
      }
    } else {
      constexpr uint32_t kIdO = idesc_bf16_f32(2 * kBM, kD, 0, 1);  // P (TMEM) x V (MN-major)
      const uint64_t dv0 = smem_desc_sw128(smem_addr(sm.v[0]), kSlotBytes, 1024);
      const uint32_t v_empty_l = cluster_addr(smem_addr(&sm.v_empty[0]), 0);
      const uint32_t v_empty_p = cluster_addr(smem_addr(&sm.v_empty[0]), 1);
      uint32_t t = 0, items = 0;
      uint32_t fix_parity = 0;  // bit s: parity of the next v_fixed phase of slot s
      while (ok) {
        const Item *ip = wait_item(sm, taken, leader, p.err);
        const int id = ip ? ip->id : -1, nk = ip ? ip->nk : 0;
        const bool fix = ip && ip->last_rows < kBN;
        release_item(item_empty_l, taken, lane);
        ++taken;
        if (!ip) {
          ok = false;
          break;
        }
        if (id < 0) break;
        if (nk == 0) continue;
        for (int j = 0; j < nk && ok; ++j, ++t) {
          const uint32_t pb = t % kSBufs, vs = t % kVSlots;
          ok = wait_all(&sm.p_full[pb], (t / kSBufs) & 1);
          // the item's first PV overwrites O: the previous item's O must have been read
          if (ok && j == 0 && items > 0) ok = wait_all(&sm.o_free, (items - 1) & 1);
          // V(t) landed in both CTAs; for an item's last tile with rows past the keys, both
          // CTAs have also zeroed them
          if (ok) ok = wait_all(&sm.v_full[vs], (t / kVSlots) & 1);
          if (ok && fix && j == nk - 1) {
            ok = __all_sync(kFull, wait_parity_cluster(&sm.v_fixed[vs], (fix_parity >> vs) & 1,
                                                       p.err));
            fix_parity ^= 1u << vs;
          }
          if (!ok) break;
          tc_fence_after_sync();
          if (elect_one()) {
            mma_pv(tmem + kOCol, tmem + 128 * pb, dv0 + vs * (kSlotBytes >> 4), kIdO, j > 0);
            commit_both(o_full_l + 8 * pb, o_full_p + 8 * pb);
            commit_both(v_empty_l + 8 * vs, v_empty_p + 8 * vs);
          }
          __syncwarp();
        }
        ++items;
      }
    }
    // every UMMA must be complete before the tensor memory is released and the pair exits,
    // also after an abort: one more commit tracks all of this warp's (the wait ignores the
    // abort bit)
    if (elect_one()) umma_commit_pair(cluster_addr(smem_addr(drain_bar), 0));
    __syncwarp();
    __all_sync(kFull, wait_own(drain_bar, 0, p.err));
  } else if (warp < kSoftmaxWarps) {
    // ------------------------------------------------------------------ softmax warps
    // Warp w owns 16 rows: TMEM lanes 16 (w / 4) .. + 16 of lane quadrant w % 4. Two threads
    // share a row (tcgen05.ld/st shape 16x32bx2): thread i and i + 16 hold its key columns
    // 0-63 and 64-127 of every tile, and combine the row max (per tile) and the row sum (per
    // item) with one shuffle. The warps never wait for each other.
    const int quad = warp & 3, lh = warp >> 2;
    const int ch = lane >> 4;                             // this thread's column half
    const int r = quad * 32 + lh * 16 + (lane & 15);      // row == TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32 + lh * 16) << 16);
    const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
    uint32_t taken = 0, g = 0;
    bool ok = true;
    // the previous item's rows, written out after the next item's first P
    bool pend = false;
    int64_t pend_row = -1;
    float pend_l = 0.f;
    uint32_t pend_g = 0;
    // O of the pending item: wait for its last PV, read this thread's half of the row,
    // release O, write the half row
    auto epilogue = [&]() -> bool {
      const float l = pend_l + __shfl_xor_sync(kFull, pend_l, 16);
      if (!__all_sync(kFull, wait_parity(&sm.o_full[pend_g % kSBufs], (pend_g / kSBufs) & 1,
                                         p.err)))
        return false;
      tc_fence_after_sync();
      uint32_t o[2][32];
#pragma unroll
      for (int c = 0; c < 2; ++c) tmem_ld16x2_32<64>(lane_addr + kOCol + 32 * c, o[c]);
#pragma unroll
      for (int c = 0; c < 2; ++c) tmem_ld_wait(o[c]);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(o_free_l);
      if (pend_row >= 0) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        uint4 *dst = reinterpret_cast<uint4 *>(p.out + pend_row * kD + 64 * ch);
        // a thread writes its own half row: one 32-byte sector per store when out allows it
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              w[k] = pack_bf16(__uint_as_float(o[c][16 * e + 2 * k]) * inv,
                               __uint_as_float(o[c][16 * e + 2 * k + 1]) * inv);
            uint4 *d = dst + c * 4 + 2 * e;
            if (p.out_32b) {
              st_global_32b(d, w);
            } else {
              d[0] = make_uint4(w[0], w[1], w[2], w[3]);
              d[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
          }
      }
      pend = false;
      return true;
    };
    while (ok) {
      const Item *ip = wait_item(sm, taken, leader, p.err);
      const int id = ip ? ip->id : -1, nk = ip ? ip->nk : 0;
      int64_t row = -1;  // output row (token x head) of this thread; -1 past the queries
      int64_t lim = -1;  // last key this row sees (-1: none)
      if (id >= 0) {
        const int64_t qi = (int64_t)ip->tok[rank] + r, Lq = ip->Lq, Lk = ip->Lk;
        if (qi < Lq) {
          row = ((int64_t)ip->q0 + qi) * p.num_q_heads + ip->hq[rank];
          lim = min(p.causal ? qi + (Lk - Lq) : Lk - 1, Lk - 1);
        }
      }
      release_item(item_empty_l, taken, lane);
      ++taken;
      if (!ip) break;
      if (id < 0) {
        if (pend) ok = epilogue();
        break;
      }
      if (nk == 0) {  // no key is visible to any row: zeros
        if (row >= 0) {
          uint4 *dst = reinterpret_cast<uint4 *>(p.out + row * kD + 64 * ch);
          for (int c = 0; c < 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < nk; ++j, ++g) {
        const uint32_t sb = g % kSBufs, s_col = 128 * sb;
        // warp-uniform results: the TMEM loads and stores below are .sync.aligned
        ok = __all_sync(kFull, wait_parity(&sm.s_full[sb], (g / kSBufs) & 1, p.err));
        if (!ok) break;
        tc_fence_after_sync();
        // last visible column of this thread's half of the tile
        const int64_t rel = lim - (int64_t)j * kBN - 64 * ch;
        const int lim_rel = (int)(rel < -1 ? -1 : (rel > 64 ? 64 : rel));

        uint32_t x[2][32];  // key columns 64 ch + 32 c + e
#pragma unroll
        for (int c = 0; c < 2; ++c) tmem_ld16x2_32<64>(lane_addr + s_col + 32 * c, x[c]);
#pragma unroll
        for (int c = 0; c < 2; ++c) tmem_ld_wait(x[c]);
        if (lim_rel < 63) {  // diagonal or last tile: columns past lim_rel are -inf
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (32 * c + e > lim_rel) x[c][e] = __float_as_uint(-INFINITY);
        }
        float mx[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          mx[c] = -INFINITY;
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            mx[c] = fmax3(mx[c], __uint_as_float(x[c][e]), __uint_as_float(x[c][e + 1]));
        }
        float m_tile = fmaxf(mx[0], mx[1]);
        m_tile = fmaxf(m_tile, __shfl_xor_sync(kFull, m_tile, 16)) * p.scale_log2;
        const float m_new = fmaxf(m_run, m_tile);
        const bool rescale = m_new > m_run + kRescaleLog2;
        float alpha = 1.f;
        if (rescale) {
          alpha = fast_exp2(m_run - m_new);
          m_run = m_new;
          l_run *= alpha;
        }
        const float neg_m = m_run == -INFINITY ? 0.f : -m_run;

        // O holds the item's tiles before this one: rescale it (never on the first tile)
        if (j > 0 && __any_sync(kFull, rescale)) {
          ok = __all_sync(kFull, wait_parity(&sm.o_full[(g - 1) % kSBufs],
                                             ((g - 1) / kSBufs) & 1, p.err));
          if (!ok) break;
          tc_fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            tmem_ld16x2_32<64>(lane_addr + kOCol + 32 * c, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st16x2_32<64>(lane_addr + kOCol + 32 * c, o);
          }
        }

        // P = 2^(s * scale_log2 - m) as bf16 pairs (two keys per column) over the first 64
        // columns of S: this warp has read all of its rows' S columns, so it may overwrite them
        const float2 nm2 = make_float2(neg_m, neg_m);
        float2 rs0 = make_float2(0.f, 0.f), rs1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
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
          tmem_st16x2_16<32>(lane_addr + s_col + 16 * c, pk);
        }
        tmem_st_wait();
        l_run += (rs0.x + rs0.y) + (rs1.x + rs1.y);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(p_full_l + sb * 8);
        // the previous item's O, now that this item's first P is on its way
        if (j == 0 && pend) {
          ok = epilogue();
          if (!ok) break;
        }
      }
      if (!ok) break;
      pend = true;
      pend_row = row;
      pend_l = l_run;
      pend_g = g - 1;
    }
  }

  // every role is done with its own copies and UMMAs; the pair leaves together (remote
  // arrivals and UMMAs touch the other CTA's memory until then)
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();
  tc_fence_after_sync();
  if (warp == kSMmaWarp) tmem_dealloc_pair(tmem, kTmemCols);
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
  // q: {64 dims, tokens, 2 halves per head}; a CTA loads its 128 rows of one head per half
  const uint64_t qdims[3] = {64, (uint64_t)a.total_q, (uint64_t)a.num_q_heads * 2};
  const uint64_t qstr[2] = {(uint64_t)a.q_tok_stride * 2, 128};
  const uint32_t qbox[3] = {64, (uint32_t)kBM, 1};
  // k, v: {64 dims, rows, 2 halves per head}; a CTA loads 64 keys x both halves of K and
  // 128 keys x its half of V
  const uint64_t kvdims[3] = {64, (uint64_t)(a.kv_rows > 0 ? a.kv_rows : 1),
                              (uint64_t)a.num_kv_heads * 2};
  const uint64_t kvstr[2] = {(uint64_t)a.kv_tok_stride * 2, 128};
  const uint32_t kbox[3] = {64, (uint32_t)kBN / 2, 2};
  const uint32_t vbox[3] = {64, (uint32_t)kBN, 1};
  if (encode_tensor_map(&qm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.q), qdims,
                        qstr, qbox, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B) != CUDA_SUCCESS ||
      encode_tensor_map(&km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.k), kvdims,
                        kvstr, kbox, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B) != CUDA_SUCCESS ||
      encode_tensor_map(&vm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.v), kvdims,
                        kvstr, vbox, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(PrefillSmem) + 1024;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // the pairs that fit on the device at once (one CTA per SM), looked up once per device
  static int max_pairs[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  int pairs = dev < 64 ? max_pairs[dev] : 0;
  if (pairs <= 0) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2 * (unsigned)(num_sms / 2));
    e = cudaOccupancyMaxActiveClusters(&pairs, prefill_kernel<G>, &cfg);
    if (e != cudaSuccess) return e;
    if (pairs <= 0) return cudaErrorInvalidConfiguration;
    if (dev < 64) max_pairs[dev] = pairs;
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
  const int64_t clusters = items < pairs ? items : pairs;
  prefill_plan_kernel<<<1, kPlanThreads, 0, stream>>>(pp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(2 * (unsigned)clusters);
  return cudaLaunchKernelEx(&cfg, prefill_kernel<G>, qm, km, vm, prm);
}

}  // namespace

bool prefill_group_supported(int group) {
  return group == 1 || group == 2 || group == 4 || group == 8;
}

cudaError_t launch_varlen_prefill(const PrefillArgs &a, int num_sms, cudaStream_t stream) {
  // token and row indices travel as 32-bit TMA coordinates and item fields
  if (a.total_q > INT32_MAX || a.kv_rows > INT32_MAX) return cudaErrorInvalidValue;
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
