// decode.cu -- paged decode attention as split-K flash-decoding (sm_103a).
//
// flash_attn_with_kvcache over the paged cache («nano-vLLM 最小化vLLM重新实现», 架构 5):
// one query token per sequence attends over its context, whose K/V rows are gathered
// through the sequence's block table. GQA: query head hq reads KV head hq / G.
//
// Work unit: sequence b, KV head h, up to two of the G query heads of h (so each K/V byte is
// read once for both heads of a Qwen3 group), and one split: the logical tokens
// [s * chunk, min((s + 1) * chunk, ctx_b)). chunk is a multiple of the 64-token tile and the
// block size a multiple of 256, so a tile never straddles a block.
//
// Persistent kernel: two CTAs per SM take units from a global queue (an atomic counter at the
// start of the workspace; units ordered split-major with the KV heads of a sequence adjacent,
// so the CTAs reading one sequence's rows run together). Every CTA draws until it draws past
// the last unit, once; the CTA whose draw is the last of those sets the counter back to
// zero, so no call has to clear it first. When there are no more units than CTAs, CTA i takes
// unit i and the counter is not used (a static grid). Per CTA, 8 consumer warps
// + 1 producer warp:
//   producer  -- takes a unit, hands it to the consumers through a 4-slot ring (the unit's
//                q rows arrive by a 1-D bulk copy into the ring slot), then streams the
//                unit's tiles: per 64-token tile it looks up block_tables[b][pos / bs] and
//                issues two TMA tensor loads (K and V, 64 tokens x 256 bytes of head h, as two
//                128-byte-swizzled planes of 64 dims) into a 3-stage ring, without stopping
//                between units. On a static grid it reads its unit's first block id before
//                the grid dependency wait and loads that tile right after it (dropped again
//                if the block table, read again, names another block);
//   consumers -- warp w owns tokens [8w, 8w + 8) of every tile; both products are warp MMAs
//                with the unit's query heads as the M rows (see the consumer section), with
//                the warp's own online softmax; at the end of a unit the 8 warp states are
//                merged through shared memory.
// With one split a unit writes bf16 output. With 2..8 splits and a static grid (one CTA per
// unit, units ordered split-minor), the splits of one (sequence, head group) form a
// thread-block cluster: each peer sends its normalised partial output and log2-sum-exp into
// rank 0's shared memory with asynchronous stores and rank 0 merges them. Otherwise a unit
// writes its partial to global memory and decode_combine_kernel merges.
//
// Algorithmic HBM bytes per (sequence, KV head, token): 256 (K) + 256 (V).
#include <math.h>

#include <algorithm>

#include "device_common.cuh"
#include "launch.h"

namespace pkv {
namespace {

constexpr int kD = 128;
constexpr int kTile = 64;
constexpr int kConsumerWarps = 8;
constexpr int kStages = 3;
constexpr unsigned int kErrWorkspace = 64u;  // PKV_DEVERR_WORKSPACE
constexpr int kRing = 4;
constexpr int kMaxCluster = 8;  // largest portable thread-block cluster
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kTileBytes = kTile * kD * 2;  // one head's K (or V) for 64 tokens: 16 KiB
constexpr int kPlaneBytes = kTileBytes / 2;  // one 64-dim half of it (a plane of 64 rows)
constexpr int kChunkRows = 8;                // a context's last tile is loaded in 8-row chunks
constexpr int kChunkBytes = kChunkRows * 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;

struct Unit {
  int32_t b, s, xg, ntiles;  // ntiles < 0: no more work
  int32_t store;             // store the sequence's new token (its last position) first
  int32_t skip;              // 1: the ring's next tile is a discarded speculative load
};

template <int GC>
struct DecodeSmem {
  uint8_t k[kStages][kTileBytes];  // must start 1024-byte aligned (128-byte swizzle atoms)
  uint8_t v[kStages][kTileBytes];
  float acc[kConsumerWarps][GC][kD];
  float m[kConsumerWarps][GC];
  float l[kConsumerWarps][GC];
  uint16_t qs[kRing][GC][kD];  // q rows of the queued units
  alignas(16) uint16_t newkv[kRing][2][kD];  // a unit's new K and V rows, bound for the pool
  Unit unit[kRing];
  alignas(16) uint32_t zero16[4];  // an all-zero ldmatrix row (q rows past GC)
  int32_t stop;  // set by the producer: an earlier wait gave up, this CTA does no work
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t unit_full[kRing];
  uint64_t newkv_full[kRing];
  uint64_t unit_empty[kRing];
  // cluster merge: in rank 0, the peers' results have landed; in a peer (clusters of more
  // than kLandSplits), rank 0's `acc` is free for them
  uint64_t cl_bar;
  uint64_t cl_ready;
};
static_assert(kMaxCluster - 1 <= kConsumerWarps, "the peers' results fit in rank 0's acc");

// Where a cluster's rank 0 receives its peers' results: with up to kLandSplits splits in an
// area of its own past the fixed layout (two CTAs still fit on an SM), else in its merge
// buffer `acc`, lent once its own merge has read it. (splits - 1) x GC x kD outputs, then
// (splits - 1) x GC log2-sum-exps, fp32.
constexpr int kLandSplits = 4;
template <int GC>
__host__ __device__ constexpr size_t land_offset() {
  return (sizeof(DecodeSmem<GC>) + 15) / 16 * 16;
}
template <int GC>
__host__ __device__ constexpr size_t smem_bytes(int cluster) {
  return (cluster >= 2 && cluster <= kLandSplits
              ? land_offset<GC>() + (size_t)(cluster - 1) * GC * (kD + 1) * sizeof(float)
              : sizeof(DecodeSmem<GC>)) + 1024;  // + 1024: the layout starts 1024-aligned
}

// Byte offset of 16-byte chunk j (dims 8j..8j+7) of token t inside a swizzled tile. The TMA
// box is {64 dims, 64 tokens, 2 halves}: half j / 8 of every token in its own 8 KiB plane of
// 128-byte rows (row t), and the 128-byte swizzle XORs the chunk index within the row with
// t mod 8, so the 8 rows of one ldmatrix (8 consecutive tokens, one chunk) hit 8 distinct
// bank groups.
__device__ __forceinline__ uint32_t tile_offset(int t, int j) {
  return (uint32_t)(((j >> 3) << 13) | (t << 7) | (((j & 7) ^ (t & 7)) << 4));
}

struct DecodeParams {
  const uint16_t *q;
  const int32_t *block_tables;
  const int32_t *context_lens;
  float *part_o;
  float *part_lse;
  uint16_t *out;
  int32_t *queue;  // next unit to hand out (the workspace's first word); nullptr: CTA i takes
                   // unit i only
  // > 0: the splits of one (sequence, head group) form a cluster of this many CTAs (CTA i
  // takes unit i, ordered split-minor); rank 0 merges them through distributed shared memory
  int32_t cluster;
  unsigned int *err;
  int64_t num_blocks;
  int64_t cap;  // longest context the table rows and the split grid can address
  int32_t table_width;
  int32_t batch;
  int32_t num_q_heads;
  int32_t group;
  int32_t head_groups;
  int32_t xgroups;  // num_kv_heads * head_groups
  int32_t block_size;
  int32_t chunk;
  int32_t splits;
  int32_t units;    // splits * batch * xgroups
  float qscale;
  // the step's new tokens (k_new == nullptr: nothing to store)
  const uint16_t *k_new;
  const uint16_t *v_new;
  int64_t k_new_stride, v_new_stride;  // elements per token
  const int64_t *slots;
  int64_t num_slots;
  uint16_t *k_cache_w;
  uint16_t *v_cache_w;
  int32_t num_kv_heads;
};

// Unit u -> (split s, sequence b, head group xg). A cluster launch orders the units
// split-minor (the splits of one sequence and head group adjacent), otherwise split-major.
__device__ __forceinline__ void unit_coords(const DecodeParams &p, int u, int &s, int &b,
                                            int &xg) {
  if (p.cluster) {
    s = u % p.splits;
    b = (u / p.splits) / p.xgroups;
    xg = (u / p.splits) % p.xgroups;
  } else {
    s = u / (p.batch * p.xgroups);
    const int r = u % (p.batch * p.xgroups);
    b = r / p.xgroups;
    xg = r % p.xgroups;
  }
}

template <int GC>
// 96 registers: warps are placed on the 4 SM sub-partitions (16K registers each), so two
// 9-warp CTAs (5 warps on some sub-partitions) fit only at <= 102 registers per thread.
__global__ void __maxnreg__(96)
    decode_split_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap,
                        const __grid_constant__ CUtensorMap kmap8,
                        const __grid_constant__ CUtensorMap vmap8, const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  DecodeSmem<GC> &sm = *reinterpret_cast<DecodeSmem<GC> *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 4) sm.zero16[threadIdx.x] = 0u;
  if (threadIdx.x == 0) {
    sm.stop = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], kConsumerWarps);
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&sm.unit_full[i], 1);
      mbar_init(&sm.newkv_full[i], 1);
      mbar_init(&sm.unit_empty[i], kConsumerWarps);
    }
    if (p.cluster) {
      mbar_init(&sm.cl_bar, p.cluster - 1);  // one arrival per peer
      mbar_init(&sm.cl_ready, 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  // in a cluster: this CTA's barriers are set up (waited for before the first remote access)
  if (p.cluster) cluster_arrive_relaxed();
  // cluster merge: this CTA's normalised output and log2-sum-exp (consumer thread g * kD + d)
  float cl_o = 0.f, cl_lse = -INFINITY;
  // Launched as a programmatic dependent of the stream's previous kernel: everything above
  // (barrier set-up) may overlap its tail; wait for that grid's completion and memory before
  // touching global memory.
  if (threadIdx.x == kConsumerWarps * 32) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    prefetch_tensormap(&kmap8);
    prefetch_tensormap(&vmap8);
  }
  // the first tile's pool row as read ahead of the wait (-1: none), and its KV head
  int32_t spec_blk = -1, spec_row = -1, spec_h = 0;
  if (!p.queue && threadIdx.x == kConsumerWarps * 32) {
    // Static grid: this CTA's unit is known now. While the previous grid finishes, warm L2
    // with its context length, and with its first tiles through a block id read ahead of the
    // wait. That read may see an old table (it is only a hint: L2 only, nothing kept in L1,
    // and every value used below is read again after the wait).
    int s, b, xg;
    unit_coords(p, blockIdx.x, s, b, xg);
    prefetch_l2(p.context_lens + b);
    const int64_t begin = (int64_t)s * p.chunk;
    if (begin < p.cap) {
      const int32_t blk =
          ld_global_cg_s32(p.block_tables + (int64_t)b * p.table_width + begin / p.block_size);
      if (blk >= 0 && blk < p.num_blocks) {
        const int in_block = (int)(begin % p.block_size);
        const int n = min(2 * kStages, min(p.chunk, p.block_size - in_block) / kTile);
        const int h = xg / p.head_groups;
        if (p.k_new == nullptr) {  // (with the store inside, the last tile waits for it)
          spec_blk = blk;
          spec_row = (int32_t)((int64_t)blk * p.block_size + in_block);
          spec_h = h;
        }
        for (int t = 0; t < n; ++t) {
          const int32_t row = (int32_t)((int64_t)blk * p.block_size + in_block + t * kTile);
          tma_prefetch_3d(&kmap, 0, row, 2 * h);
          tma_prefetch_3d(&vmap, 0, row, 2 * h);
        }
      }
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the merge kernel that follows may be scheduled now: it waits for this grid's completion
  // (and its memory) before reading anything
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
    const uint64_t policy = policy_evict_first();
    uint32_t pushed = 0, tiles = 0;
    bool ok = true;
    int static_next = blockIdx.x;  // without a queue: unit blockIdx.x, then nothing
    uint32_t newkv_par = 0;        // bit s: parity of newkv_full[s]'s next phase
    bool newkv_pending = false;    // new-token rows on their way into shared memory
    int newkv_slot = 0;
    bool first_unit = true;  // the abort bit is read with the first unit's loads
    // The work counter (queued grid). Every CTA draws until it draws past the last unit, once:
    // those draws return units .. units + grid - 1, so the CTA with the highest one is the
    // last to touch the counter, and it sets the counter back to zero for the next call. From
    // a zeroed counter a CTA's first draw is below units + grid: anything else (or a draw
    // below zero) means the workspace's counter was not zero on entry.
    bool first_draw = true, past_end = false;
    int last_rows = kTile;  // keys in the current unit's last tile
    auto draw = [&]() -> int {
      const int u = atomicAdd(p.queue, 1);
      if (first_draw) {
        first_draw = false;
        if (u < 0 || u >= p.units + (int)gridDim.x) record_error(p.err, kErrWorkspace);
      }
      if (u < 0 || u >= p.units) {
        past_end = true;
        if (u == p.units + (int)gridDim.x - 1) atomicExch(p.queue, 0);
      }
      return u;
    };
    // The first tile's K and V are loaded at once with the block id read ahead of the wait;
    // once the block table is read again, the tile is kept if the id still holds, else the
    // consumers discard it (Unit::skip) and the tile is loaded again.
    bool spec_pending = false;
    if (spec_row >= 0) {
      mbar_arrive_expect_tx(&sm.full[0], 2 * kTileBytes);
      tma_load_3d(sm.k[0], &kmap, &sm.full[0], 0, spec_row, 2 * spec_h, policy);
      tma_load_3d(sm.v[0], &vmap, &sm.full[0], 0, spec_row, 2 * spec_h, policy);
      tiles = 1;
      spec_pending = true;
    }
    while (ok) {
      // next unit with work (or one that must write zeros); ntiles < 0 ends the walk
      Unit un{0, 0, 0, -1, 0, 0};
      int32_t first_blk = -1;  // block id of the unit's first tile
      int first_it = 0;        // tiles of the unit already loaded
      while (true) {
        int u;
        if (p.queue) {
          u = draw();
        } else {
          u = static_next;
          static_next = p.units;
        }
        if (u < 0 || u >= p.units) break;
        int s, b, xg;
        unit_coords(p, u, s, b, xg);
        // the first tile's block id does not depend on the context length: both loads are in
        // flight together (a unit that starts past the table's end reads no entry)
        const int64_t begin = (int64_t)s * p.chunk;
        // an earlier wait gave up somewhere: end the walk (in a cluster the CTA still takes
        // part in the cluster's barriers)
        const uint32_t err_now =
            first_unit && p.err ? (uint32_t)ld_global_s32(reinterpret_cast<const int32_t *>(p.err)) : 0u;
        int64_t L;
        if (begin < p.cap) {
          L = ld_global_s32(p.context_lens + b);
          first_blk = ld_global_s32(p.block_tables + (int64_t)b * p.table_width +
                                    begin / p.block_size);
        } else {
          L = ld_global_s32(p.context_lens + b);
        }
        if (first_unit) {
          first_unit = false;
          if (err_now & kErrTimeout) {
            sm.stop = 1;
            break;
          }
        }
        if (L < 0 || L > p.cap) {
          if (s == 0 && xg == 0) record_error(p.err, 4u /* CONTEXT_RANGE */);
          L = L < 0 ? 0 : p.cap;
        }
        if (begin < L) {
          const int64_t end = min(L, begin + p.chunk);
          // the unit that reads position L - 1 stores the new token there first (only one
          // unit per KV head reads it: the launcher takes this path with one head group)
          un = Unit{b, s, xg, (int)((end - begin + kTile - 1) / kTile),
                    p.k_new != nullptr && end == L ? 1 : 0, 0};
          last_rows = (int)(end - begin - (int64_t)(un.ntiles - 1) * kTile);
          if (spec_pending) {
            if (first_blk == spec_blk) first_it = 1;
            else un.skip = 1;
            spec_pending = false;
          }
          break;
        }
        if (p.cluster || (L == 0 && s == 0 && p.splits == 1)) {
          // nothing to read: zeros (empty context), or in a cluster no result (the unit
          // still leaves its -inf log2-sum-exp for the merge)
          un = Unit{b, s, xg, 0, 0, spec_pending ? 1 : 0};
          spec_pending = false;
          break;
        }
      }
      const int slot = pushed % kRing;
      if (pushed >= kRing &&
          !wait_parity(&sm.unit_empty[slot], ((pushed / kRing) - 1) & 1, p.err)) {
        ok = false;
        break;
      }
      sm.unit[slot] = un;
      ++pushed;
      if (un.ntiles < 0) {
        mbar_arrive(&sm.unit_full[slot]);
        break;
      }
      const int h = un.xg / p.head_groups;
      const int hq0 = h * p.group + (un.xg % p.head_groups) * GC;
      mbar_arrive_expect_tx(&sm.unit_full[slot], GC * kD * 2);
      bulk_copy_g2s(sm.qs[slot], p.q + ((int64_t)un.b * p.num_q_heads + hq0) * kD, GC * kD * 2,
                    &sm.unit_full[slot]);
      // the unit that reads the context's last position brings the new token's K and V rows
      // of its head into shared memory now (the pool write happens before its last tile)
      uint16_t *store_dst = nullptr, *store_dst_v = nullptr;
      if (un.store) {
        const int64_t sl = p.slots[un.b];
        if (sl >= p.num_slots) record_error(p.err, 1u /* SLOT_RANGE */);
        if (sl >= 0 && sl < p.num_slots) {
          store_dst = p.k_cache_w + (sl * p.num_kv_heads + h) * kD;
          store_dst_v = p.v_cache_w + (sl * p.num_kv_heads + h) * kD;
          mbar_arrive_expect_tx(&sm.newkv_full[slot], 2 * kD * 2);
          bulk_copy_g2s(sm.newkv[slot][0], p.k_new + un.b * p.k_new_stride + h * kD, kD * 2,
                        &sm.newkv_full[slot]);
          bulk_copy_g2s(sm.newkv[slot][1], p.v_new + un.b * p.v_new_stride + h * kD, kD * 2,
                        &sm.newkv_full[slot]);
          newkv_pending = true;
          newkv_slot = slot;
        }
      }
      const int32_t *table = p.block_tables + (int64_t)un.b * p.table_width;
      const int tok_begin = un.s * p.chunk;
      for (int it = first_it; it < un.ntiles; ++it, ++tiles) {
        const int stage = tiles % kStages;
        if (tiles >= kStages && !wait_parity(&sm.empty[stage], ((tiles / kStages) - 1) & 1, p.err)) {
          ok = false;
          break;
        }
        if (store_dst && it == un.ntiles - 1) {
          // This tile holds the context's last position: the new token's rows must be in the
          // pool before its TMA load. They arrived in shared memory at the unit's start; copy
          // them out with the bulk engine and wait for the writes (all in the async proxy, so
          // the load below is ordered after them).
          if (!wait_parity(&sm.newkv_full[slot], (newkv_par >> slot) & 1, p.err)) {
            ok = false;
            break;
          }
          newkv_par ^= 1u << slot;
          newkv_pending = false;
          bulk_copy_s2g(store_dst, sm.newkv[slot][0], kD * 2);
          bulk_copy_s2g(store_dst_v, sm.newkv[slot][1], kD * 2);
          bulk_commit();
          bulk_wait_all();
        }
        const int pos = tok_begin + it * kTile;
        const int64_t blk = it == 0 ? first_blk : table[pos / p.block_size];
        int32_t row;
        if (blk < 0 || blk >= p.num_blocks) {
          record_error(p.err, 2u /* BLOCK_RANGE */);
          row = -2 * kTile;  // wholly outside the pool: TMA fills zeros, nothing is read
        } else {
          row = (int32_t)(blk * p.block_size + pos % p.block_size);
        }
        const int rows_here = it == un.ntiles - 1 ? last_rows : kTile;
        if (rows_here >= kTile || row < 0) {
          mbar_arrive_expect_tx(&sm.full[stage], 2 * kTileBytes);
          tma_load_3d(sm.k[stage], &kmap, &sm.full[stage], 0, row, 2 * h, policy);
          tma_load_3d(sm.v[stage], &vmap, &sm.full[stage], 0, row, 2 * h, policy);
        } else {
          // the unit's last tile ends inside the tile: only its 8-row chunks that hold keys
          // (the consumers mask the rows past the context, whatever shared memory holds)
          const int chunks = (rows_here + kChunkRows - 1) / kChunkRows;
          mbar_arrive_expect_tx(&sm.full[stage], (uint32_t)(chunks * 4 * kChunkBytes));
          for (int c = 0; c < chunks; ++c)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const int off = hf * kPlaneBytes + c * kChunkBytes;
              tma_load_3d(sm.k[stage] + off, &kmap8, &sm.full[stage], 0, row + kChunkRows * c,
                          2 * h + hf, policy);
              tma_load_3d(sm.v[stage] + off, &vmap8, &sm.full[stage], 0, row + kChunkRows * c,
                          2 * h + hf, policy);
            }
        }

      }
    }
    // a CTA that stopped early (an abort, a wait that gave up) still draws past the last unit
    // once, so that the counter goes back to zero
    if (p.queue)
      while (!past_end) draw();
    // keep the CTA alive until every copy it issued has landed (also after an abort: these
    // waits ignore the abort bit; `tiles` and `pushed` count only issued copies)
    bool drained = true;
    if (newkv_pending) drained = wait_own(&sm.newkv_full[newkv_slot], (newkv_par >> newkv_slot) & 1, p.err);
    for (uint32_t t = tiles > kStages ? tiles - kStages : 0; drained && t < tiles; ++t)
      drained = wait_own(&sm.full[t % kStages], (t / kStages) & 1, p.err);
    for (uint32_t k = pushed > kRing ? pushed - kRing : 0; drained && k < pushed; ++k)
      drained = wait_own(&sm.unit_full[k % kRing], (k / kRing) & 1, p.err);
    }
    if (!p.cluster) return;
    __syncwarp();
  } else {

  // -------------------------------------------------------------------- consumers
  // Warp w owns tokens [8w, 8w + 8) of every 64-token tile; both products run as warp-level
  // MMAs with the unit's query heads as the M rows (GC of 16 used):
  //   S   (16 heads x 8 tokens) = Q (16 x 128) K^T        m16n8k16, 8 steps over the dims
  //   O^T (16 dims x 8 heads)  += V^T (16 x 8 tokens) P^T  m16n8k8, 8 blocks of 16 dims
  // Lane l = 4 gq + tq holds S for head gq and tokens 2tq, 2tq + 1, which is exactly its
  // share of the P^T operand of the second product: P stays in registers (rounded to bf16,
  // and l sums the rounded values). Its O^T accumulator holds heads 2tq and 2tq + 1.
  const int gq = lane >> 2, tq = lane & 3;
  const int tok = warp * 8 + 2 * tq;  // tile-relative token of S column 2tq
  // ldmatrix row addresses: lanes 8i..8i+7 give matrix i of load j = dims chunk 4j + i of
  // tokens 8w..8w+7
  uint32_t off_ld[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) off_ld[j] = tile_offset(warp * 8 + (lane & 7), 4 * j + (lane >> 3));
  const uint32_t k_base = smem_addr(sm.k[0]), v_base = smem_addr(sm.v[0]);
  // q: ldmatrix row (lane & 7) = head, matrix (lane >> 3) = dims chunk; heads past GC read zeros
  const bool q_row = (lane & 7) < GC;
  const uint32_t q_zero = smem_addr(sm.zero16);

  // Every decision to leave the unit loop is taken by all 8 consumer warps together (a
  // barrier reduction), so no warp can be left waiting in a merge barrier.
  uint32_t taken = 0, tiles = 0;
  while (true) {
    const int slot = taken % kRing;
    const bool got = wait_parity(&sm.unit_full[slot], (taken / kRing) & 1, p.err);
    if (barrier_or(3, kConsumerWarps * 32, !got)) break;
    const Unit un = sm.unit[slot];
    ++taken;
    if (un.ntiles < 0) break;
    const int h = un.xg / p.head_groups;
    const int hq0 = h * p.group + (un.xg % p.head_groups) * GC;
    // q's A fragments, held in registers for the unit: load j gives dims [32j, 32j + 32) as
    // a0, a2 of k-step 2j and a0, a2 of k-step 2j + 1 (rows 8-15, a1 and a3, are zero)
    uint32_t qa[4][4];
    {
      const uint32_t q_base =
          q_row ? smem_addr(&sm.qs[slot][lane & 7][8 * (lane >> 3)]) : q_zero;
      const uint32_t q_step = q_row ? 64u : 0u;  // 4 chunks of 16 bytes per load
#pragma unroll
      for (int j = 0; j < 4; ++j) ldsm_x4(q_base + j * q_step, qa[j]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.unit_empty[slot]);

    int64_t L = p.context_lens[un.b];
    L = L < 0 ? 0 : (L > p.cap ? p.cap : L);
    const int tok_begin = un.s * p.chunk;
    const int tok_end = (int)min(L, (int64_t)tok_begin + p.chunk);

    float m_run = -INFINITY;  // running maximum of head gq (the same in the lane's quad)
    float l_run = 0.f;        // this lane's share of head gq's sum
    float acc[8][4];          // O^T: dims 16m + gq (+8) x heads 2tq, 2tq + 1
#pragma unroll
    for (int m = 0; m < 8; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;

    bool ok = true;
    if (un.skip) {  // a speculative load of the first tile that did not hold: let it land, drop it
      const int stage = tiles % kStages;
      ok = __all_sync(kFull, wait_parity(&sm.full[stage], (tiles / kStages) & 1, p.err));
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(&sm.empty[stage]);
      ++tiles;
    }
    for (int it = 0; ok && it < un.ntiles; ++it, ++tiles) {
      const int stage = tiles % kStages;
      // warp-uniform: the loop body uses warp-wide MMAs and shuffles
      if (!__all_sync(kFull, wait_parity(&sm.full[stage], (tiles / kStages) & 1, p.err))) {
        ok = false;
        break;
      }
      const uint32_t kt = k_base + stage * kTileBytes;
      const uint32_t vt = v_base + stage * kTileBytes;
      const int n_valid = tok_end - (tok_begin + it * kTile);  // >= 1; < 64 only in a last tile

      // ---- S = Q K^T for the warp's 8 tokens (two accumulators: half the dependency chain)
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // dims [32j, 32j + 32): two k-steps
        uint32_t kb[4];
        ldsm_x4(kt + off_ld[j], kb);  // token rows: dims chunks 4j .. 4j + 3
        mma_bf16_16816(s0, qa[j][0], 0u, qa[j][1], 0u, kb[0], kb[1]);
        mma_bf16_16816(s1, qa[j][2], 0u, qa[j][3], 0u, kb[2], kb[3]);
      }
      uint32_t vb[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) ldsm_x4_trans(vt + off_ld[j], &vb[4 * j]);

      // ---- online softmax (log2 domain); heads past GC and tokens past the context drop out
      float sa = (s0[0] + s1[0]) * p.qscale;
      float sb = (s0[1] + s1[1]) * p.qscale;
      if (gq >= GC) sa = sb = -INFINITY;
      if (n_valid < kTile) {
        if (tok >= n_valid) sa = -INFINITY;
        if (tok + 1 >= n_valid) sb = -INFINITY;
        // their V rows may hold anything (0 * NaN would poison the sums): zero them
        const uint32_t vmask = (tok < n_valid ? 0x0000ffffu : 0u) | (tok + 1 < n_valid ? 0xffff0000u : 0u);
#pragma unroll
        for (int c = 0; c < 16; ++c) vb[c] &= vmask;
      }
      float mx = fmaxf(sa, sb);
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
      if (__any_sync(kFull, mx > m_run)) {
        const float m_new = fmaxf(m_run, mx);
        const float alpha = m_new == -INFINITY ? 1.f : fast_exp2(m_run - m_new);
        l_run *= alpha;
        m_run = m_new;
        // the accumulator's heads 2tq and 2tq + 1 live in quads 2tq and 2tq + 1
        const float a_lo = __shfl_sync(kFull, alpha, 8 * tq);
        const float a_hi = __shfl_sync(kFull, alpha, 8 * tq + 4);
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          acc[m][0] *= a_lo;
          acc[m][1] *= a_hi;
          acc[m][2] *= a_lo;
          acc[m][3] *= a_hi;
        }
      }
      float pa = 0.f, pb = 0.f;
      if (m_run != -INFINITY) {
        pa = fast_exp2(sa - m_run);
        pb = fast_exp2(sb - m_run);
      }
      const uint32_t pf = pack_bf16x2(pa, pb);
      l_run += bf16_lo(pf) + bf16_hi(pf);

      // ---- O^T += V^T P^T
#pragma unroll
      for (int m = 0; m < 8; ++m) mma_bf16_1688(acc[m], vb[2 * m], vb[2 * m + 1], pf);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[stage]);
    }

    // ---- merge: the quad's shares of l, then the 8 warps through shared memory
    l_run += __shfl_xor_sync(kFull, l_run, 1);
    l_run += __shfl_xor_sync(kFull, l_run, 2);
    if (tq == 0 && gq < GC) {
      sm.m[warp][gq] = m_run;
      sm.l[warp][gq] = l_run;
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int hh = 2 * tq + e;
      if (hh < GC) {
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          sm.acc[warp][hh][16 * m + gq] = acc[m][e];
          sm.acc[warp][hh][16 * m + gq + 8] = acc[m][2 + e];
        }
      }
    }
    if (barrier_or(1, kConsumerWarps * 32, !ok)) break;  // a wait gave up: stop together
    const int g = threadIdx.x / kD;
    const int d = threadIdx.x % kD;
    if (g < GC) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm.m[w][g]);
      float o = 0.f, lse = -INFINITY;
      if (M != -INFINITY) {
        float lsum = 0.f, osum = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float f = fast_exp2(sm.m[w][g] - M);
          lsum = fmaf(sm.l[w][g], f, lsum);
          osum = fmaf(sm.acc[w][g][d], f, osum);
        }
        // lsum >= 1 (the warp holding the maximum contributes 2^0): the approximate division
        // and log2 err far below one bf16 rounding of the result
        o = __fdividef(osum, lsum);
        lse = M + __log2f(lsum);
      }
      const int64_t row = (int64_t)un.b * p.num_q_heads + hq0 + g;
      if (p.cluster) {  // merged by the cluster's rank 0 at the end
        cl_o = o;
        cl_lse = lse;  // -inf when the unit had no keys
      } else if (p.splits == 1 || (un.s == 0 && tok_end == L)) {
        // the unit holds the whole context: the output itself (the merge kernel skips rows
        // whose context fits one split)
        p.out[row * kD + d] = bf16_bits_rn(o);
      } else {
        p.part_o[(row * p.splits + un.s) * kD + d] = o;
        if (d == 0) p.part_lse[row * p.splits + un.s] = lse;
      }
    }
    if (!p.queue) break;  // a static grid gives each CTA one unit: nothing follows
    named_barrier_sync(2, kConsumerWarps * 32);  // merge buffer free for the next unit
  }
  }
  if (!p.cluster) return;
  // ---------------------------------------------------------------- cluster merge
  // The CTAs of the cluster are the splits of one sequence and head group. Each peer sends
  // its result into rank 0's landing area (for more than kLandSplits splits, rank 0's merge
  // buffer, which rank 0 lends once its own merge has read it) with asynchronous stores
  // counted on rank 0's barrier and leaves; rank 0 waits for the bytes, merges and writes the
  // output. (Rank 0 never reads a peer's memory, so the peers need not wait for it to
  // finish.) The waits below ignore the abort bit: every CTA reaches this point (its other
  // waits are bounded), rank 0 always lends the buffer and every peer always sends, so no
  // store lands in a CTA that has left.
  cluster_wait();  // every CTA's barriers are set up
  if (threadIdx.x >= GC * kD) return;
  const uint32_t rank = cluster_ctarank();
  const bool lend = p.cluster > kLandSplits;
  float *land_o = lend ? &sm.acc[0][0][0]  // peer r + 1's outputs at [r][g][d], then its lses
                       : reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(&sm) +
                                                   land_offset<GC>());
  float *land_lse = land_o + (size_t)(p.cluster - 1) * GC * kD;
  const int g = threadIdx.x / kD, d = threadIdx.x % kD;
  if (rank != 0) {
    if (lend && !wait_own(&sm.cl_ready, 0, p.err)) return;
    const uint32_t bar = cluster_addr(smem_addr(&sm.cl_bar), 0);
    if (threadIdx.x == 0) mbar_arrive_expect_tx_remote(bar, GC * (kD + 1) * sizeof(float));
    const int r = (int)rank - 1;
    st_async_f32(cluster_addr(smem_addr(land_o + ((size_t)r * GC + g) * kD + d), 0), cl_o, bar);
    if (d == 0) st_async_f32(cluster_addr(smem_addr(land_lse + r * GC + g), 0), cl_lse, bar);
    return;
  }
  if (lend) {
    // every merging thread has read `acc` (its values are in registers): lend it to the peers
    named_barrier_sync(2, GC * kD);
    if (threadIdx.x == 0)
      for (int r = 1; r < p.cluster; ++r)
        mbar_arrive_remote(cluster_addr(smem_addr(&sm.cl_ready), r));
  }
  if (!wait_own(&sm.cl_bar, 0, p.err)) return;
  float M = cl_lse;
  for (int r = 0; r < p.cluster - 1; ++r) M = fmaxf(M, land_lse[r * GC + g]);
  float acc = 0.f, wsum = 0.f;
  if (M != -INFINITY) {
    const float w0 = fast_exp2(cl_lse - M);  // 0 for a split with no keys
    wsum = w0;
    acc = w0 * cl_o;
    for (int r = 0; r < p.cluster - 1; ++r) {
      const float wgt = fast_exp2(land_lse[r * GC + g] - M);
      wsum += wgt;
      acc = fmaf(wgt, land_o[((size_t)r * GC + g) * kD + d], acc);
    }
  }
  const int unit0 = blockIdx.x;  // rank 0 holds split 0
  const int b = (unit0 / p.splits) / p.xgroups, xg = (unit0 / p.splits) % p.xgroups;
  const int h = xg / p.head_groups;
  const int64_t row = (int64_t)b * p.num_q_heads + h * p.group + (xg % p.head_groups) * GC + g;
  if (!sm.stop) p.out[row * kD + d] = bf16_bits_rn(wsum > 0.f ? acc / wsum : 0.f);
}

// One warp per (sequence, query head): out = sum_s 2^(lse_s - lse) o_s over the sequence's
// splits, lse = log2 sum_s 2^lse_s. A sequence with no token gets zeros; one whose context
// fits one split was written by the split kernel.
__global__ void __launch_bounds__(128)
    decode_combine_kernel(const float *__restrict__ part_o, const float *__restrict__ part_lse,
                          const int32_t *__restrict__ context_lens, int32_t batch,
                          int32_t num_q_heads, int32_t chunk, int32_t splits, int64_t cap,
                          uint16_t *__restrict__ out, const unsigned int *err) {
  // the stream's next kernel (the next call's split kernel) may be scheduled now: it waits
  // for this grid's completion before it touches global memory
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // launched as a programmatic dependent of the split kernel: wait until that grid has
  // completed and its partial results are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (aborted(err)) return;  // an earlier wait gave up: the partials are not complete
  const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= (int64_t)batch * num_q_heads) return;
  const int lane = threadIdx.x & 31;
  const int b = (int)(row / num_q_heads);
  int64_t L = context_lens[b];
  L = L < 0 ? 0 : (L > cap ? cap : L);
  const int ns = (int)((L + chunk - 1) / chunk);
  if (ns == 1) return;  // one split: the split kernel wrote this row itself
  const float *lse = part_lse + row * splits;
  float M = -INFINITY;
  for (int s = lane; s < ns; s += 32) M = fmaxf(M, lse[s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < ns; ++s) {
      const float wgt = fast_exp2(lse[s] - M);
      const float4 o4 = *reinterpret_cast<const float4 *>(part_o + (row * splits + s) * kD + 4 * lane);
      wsum += wgt;
      acc.x = fmaf(wgt, o4.x, acc.x);
      acc.y = fmaf(wgt, o4.y, acc.y);
      acc.z = fmaf(wgt, o4.z, acc.z);
      acc.w = fmaf(wgt, o4.w, acc.w);
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const uint32_t lo = (uint32_t)bf16_bits_rn(acc.x * inv) | ((uint32_t)bf16_bits_rn(acc.y * inv) << 16);
  const uint32_t hi = (uint32_t)bf16_bits_rn(acc.z * inv) | ((uint32_t)bf16_bits_rn(acc.w * inv) << 16);
  *reinterpret_cast<uint2 *>(out + row * kD + 4 * lane) = make_uint2(lo, hi);
}

template <int GC>
cudaError_t launch_split(const CUtensorMap &km, const CUtensorMap &vm, const CUtensorMap &km8,
                         const CUtensorMap &vm8, const DecodeParams &prm, int num_sms,
                         cudaStream_t stream) {
  const size_t smem = smem_bytes<GC>(prm.cluster);
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<GC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_bytes<GC>(kLandSplits));
    if (e != cudaSuccess) return e;
    // all of the unified L1/shared storage as shared memory, so two CTAs fit on an SM
    e = cudaFuncSetAttribute(decode_split_kernel<GC>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const int64_t ctas = std::min<int64_t>((int64_t)num_sms * 2, prm.units);
  // a programmatic dependent of the stream's previous kernel: its launch and barrier set-up
  // overlap that kernel's tail (it waits for the grid before reading anything)
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (prm.cluster) {  // one CTA per unit, the splits of a (sequence, head group) in a cluster
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)prm.cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, decode_split_kernel<GC>, km, vm, km8, vm8, prm);
}

}  // namespace

DecodePlan plan_decode(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t max_context_len, int32_t num_splits, int num_sms) {
  DecodePlan p{};
  const int group = num_q_heads / num_kv_heads;
  p.heads_per_cta = (group % 2 == 0) ? 2 : 1;
  p.head_groups = group / p.heads_per_cta;
  const int64_t max_ctx = max_context_len > 0 ? max_context_len : 1;
  const int64_t max_tiles = (max_ctx + kTile - 1) / kTile;
  if (num_splits > 0) {
    const int64_t S = num_splits < max_tiles ? num_splits : max_tiles;
    const int64_t per = (max_ctx + S - 1) / S;
    p.chunk = (int32_t)((per + kTile - 1) / kTile * kTile);
  } else {
    // At most 16 tiles per unit (a CTA streams its unit through a 3-tile ring, so long
    // units cap the bandwidth of a skewed batch; the work queue balances short ones), or 32
    // once there are at least 8 units per SM: then the queue hides the long units' tail, and
    // one split fewer saves the partial results and the merge (Qwen3 batch, 256 contexts up
    // to 2048 tokens: 1 split 178.5 us per call against 179.9 us with 2). Below that, more
    // splits give more CTAs for a small batch, but every CTA past one per SM shares an SM,
    // and a unit's fixed costs (its first tile's latency, the merges) do not shrink.
    // Measured on batches 1..64 at 1024 tokens, the best split count is the largest that
    // keeps its splits within one cluster and the grid within about 1.7 CTAs per SM, or
    // within one CTA per SM for clusters of more than 4 (larger clusters do not all fit at
    // once when SMs hold two CTAs).
    const int64_t units = (int64_t)batch * num_kv_heads * p.head_groups;
    const int64_t max_unit_tiles = units >= 8LL * num_sms ? 32 : 16;
    int64_t S = (max_tiles + max_unit_tiles - 1) / max_unit_tiles;
    while (S < max_tiles && S < kMaxCluster &&
           units * (S + 1) <= (S + 1 > 4 ? (int64_t)num_sms : (int64_t)num_sms * 17 / 10))
      ++S;
    const int64_t per = (max_ctx + S - 1) / S;
    p.chunk = (int32_t)((per + kTile - 1) / kTile * kTile);
  }
  p.splits = (int32_t)((max_ctx + p.chunk - 1) / p.chunk);
  const size_t partials =
      p.splits > 1 ? (size_t)batch * num_q_heads * p.splits * (kD + 1) * sizeof(float) : 0;
  p.workspace_bytes = kDecodeQueueBytes + (partials + 15) / 16 * 16;  // the counters first
  return p;
}

cudaError_t launch_paged_decode(const DecodeArgs &a, const DecodePlan &p, cudaStream_t stream) {
  // TMA views of the two pools: {64 dims, num_blocks * block_size rows, 2 * Hkv half-heads}
  // (the half-head stride, 128 bytes, is the innermost of the two): a tile lands as two
  // planes, one per half of the head dimension. The second pair of views moves 8 rows of one
  // half: a context's last tile is loaded only as far as it holds keys.
  CUtensorMap km, vm, km8, vm8;
  const uint64_t rows = (uint64_t)a.num_blocks * a.block_size;
  const uint64_t dims[3] = {64, rows, (uint64_t)a.num_kv_heads * 2};
  const uint64_t strides[2] = {(uint64_t)a.num_kv_heads * kD * 2, 128};
  const uint32_t box[3] = {64, kTile, 2};
  const uint32_t box8[3] = {64, kChunkRows, 1};
  if (encode_tensor_map(&km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.k_cache),
                        dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B) != CUDA_SUCCESS ||
      encode_tensor_map(&vm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.v_cache),
                        dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B) != CUDA_SUCCESS ||
      encode_tensor_map(&km8, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.k_cache),
                        dims, strides, box8, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B) != CUDA_SUCCESS ||
      encode_tensor_map(&vm8, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.v_cache),
                        dims, strides, box8, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  uint8_t *ws = static_cast<uint8_t *>(a.workspace);
  float *const part_base = reinterpret_cast<float *>(ws + kDecodeQueueBytes);  // after the counter
  DecodeParams prm{};
  prm.q = static_cast<const uint16_t *>(a.q);
  prm.block_tables = a.block_tables;
  prm.context_lens = a.context_lens;
  prm.part_o = p.splits > 1 ? part_base : nullptr;
  prm.part_lse = p.splits > 1 ? prm.part_o + (size_t)a.batch * a.num_q_heads * p.splits * kD
                              : nullptr;
  prm.out = static_cast<uint16_t *>(a.out);
  prm.queue = reinterpret_cast<int32_t *>(ws);
  prm.err = a.err;
  prm.num_blocks = a.num_blocks;
  prm.cap = std::min((int64_t)a.table_width * a.block_size, (int64_t)p.splits * p.chunk);
  prm.table_width = a.table_width;
  prm.batch = a.batch;
  prm.num_q_heads = a.num_q_heads;
  prm.group = a.num_q_heads / a.num_kv_heads;
  prm.head_groups = p.head_groups;
  prm.xgroups = a.num_kv_heads * p.head_groups;
  prm.block_size = a.block_size;
  prm.chunk = p.chunk;
  prm.splits = p.splits;
  const int64_t units = (int64_t)p.splits * a.batch * prm.xgroups;
  // the work counter runs to units + grid size - 1 (an int): keep that in range
  if (units + 2 * (int64_t)a.num_sms > INT32_MAX) return cudaErrorInvalidValue;
  prm.units = (int32_t)units;
  prm.qscale = a.scale * kLog2e;
  prm.num_kv_heads = a.num_kv_heads;
  if (a.k_new) {
    if (p.head_groups == 1) {  // each KV head's last position is read by one unit: fused
      prm.k_new = static_cast<const uint16_t *>(a.k_new);
      prm.v_new = static_cast<const uint16_t *>(a.v_new);
      prm.k_new_stride = a.k_new_stride;
      prm.v_new_stride = a.v_new_stride;
      prm.slots = a.slot_mapping;
      prm.num_slots = a.num_slots;
      prm.k_cache_w = static_cast<uint16_t *>(const_cast<void *>(a.k_cache));
      prm.v_cache_w = static_cast<uint16_t *>(const_cast<void *>(a.v_cache));
    } else {  // several CTAs read one head's rows: store first, as a kernel of its own
      cudaError_t e = launch_kv_store(a.k_new, a.k_new_stride, a.v_new, a.v_new_stride,
                                      a.slot_mapping, a.batch, const_cast<void *>(a.k_cache),
                                      const_cast<void *>(a.v_cache), a.num_slots,
                                      (int64_t)a.num_kv_heads * kD, a.err, a.num_sms, stream);
      if (e != cudaSuccess) return e;
    }
  }

  // With no more units than CTAs each CTA takes unit blockIdx.x and the counters are not
  // used. Then, with 2 to kMaxCluster splits, the splits of one (sequence, head group) run as
  // one thread-block cluster and merge in distributed shared memory: no partials in global
  // memory and no merge kernel. With the queue the kernel leaves the counters at zero
  // itself, so the call enqueues nothing before it (the kernel follows the previous one as a
  // programmatic dependent).
  const bool queued = (int64_t)a.num_sms * 2 < units;
  cudaError_t e = cudaSuccess;
  if (!queued) prm.queue = nullptr;
  if (e != cudaSuccess) return e;
  prm.cluster = !queued && p.splits >= 2 && p.splits <= kMaxCluster ? p.splits : 0;
  e = p.heads_per_cta == 2 ? launch_split<2>(km, vm, km8, vm8, prm, a.num_sms, stream)
                           : launch_split<1>(km, vm, km8, vm8, prm, a.num_sms, stream);
  if (e != cudaSuccess || p.splits == 1 || prm.cluster) return e;
  const int64_t rows_out = (int64_t)a.batch * a.num_q_heads;
  // programmatic dependent launch: the merge grid is set up while the split kernel runs
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)((rows_out + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_combine_kernel, (const float *)prm.part_o,
                            (const float *)prm.part_lse, a.context_lens, a.batch, a.num_q_heads,
                            p.chunk, p.splits, prm.cap, static_cast<uint16_t *>(a.out),
                            (const unsigned int *)a.err);
}

}  // namespace pkv
