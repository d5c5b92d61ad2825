// block_manager.cpp -- the host-side owner of the paged KV pool's blocks, with prefix caching.
//
// «nano-vLLM 最小化vLLM重新实现», 架构 3 (块管理器): the pool is cut into fixed-size blocks
// (256 tokens by default); each block carries a reference count and a hash so that blocks
// holding the same prefix can be shared; allocate() first looks for cached blocks whose hash
// matches and only takes new blocks for the rest; block hashes are xxhash over the block's
// token ids; preemption frees a sequence's blocks. The per-sequence block list is the page
// table of «企业官网建设流程全解析 (Nano-vLLM 指南)» §2.2, and reusing the cached prefix so
// that only the rest is computed is its §4.4.
//
// Readings (the pages give the idea, not the rules):
//   - A block is hashed only when it is full. Its hash is XXH64 (seed 0) over the previous
//     block's hash (8 bytes, little-endian; absent for the first block) followed by the
//     block's token ids (int32, little-endian), so equal hashes mean equal prefixes up to and
//     including the block. A hash hit is accepted only if the cached block's token ids are
//     equal too (a collision guard).
//   - Once a block of a new sequence misses, every later block of that sequence is new.
//   - Free blocks are handed out first-in first-out, starting from 0, 1, 2, ... A freed block
//     keeps its hash and tokens (it can still be hit) until it is handed out again; then its
//     hash entry is dropped.
//   - allocate() needs as many free blocks as the sequence has blocks (hits may use fewer),
//     and changes nothing when they are not there.
//   - After a token is appended (the sequence now has n tokens): if position n - 1 starts a
//     block, a new block is taken; if n fills a block, that block is hashed and registered.
//
// The XXH64 routine follows the published xxHash specification (64-bit variant).
#include <stdint.h>
#include <string.h>

#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv.h"

namespace {

// ---------------------------------------------------------------------------- XXH64
constexpr uint64_t kP1 = 0x9E3779B185EBCA87ull;
constexpr uint64_t kP2 = 0xC2B2AE3D27D4EB4Full;
constexpr uint64_t kP3 = 0x165667B19E3779F9ull;
constexpr uint64_t kP4 = 0x85EBCA77C2B2AE63ull;
constexpr uint64_t kP5 = 0x27D4EB2F165667C5ull;

inline uint64_t rotl(uint64_t x, int r) { return (x << r) | (x >> (64 - r)); }
// explicit little-endian reads, whatever the host's byte order
inline uint64_t le64(const uint8_t *p) {
  uint64_t v = 0;
  for (int i = 7; i >= 0; --i) v = (v << 8) | p[i];
  return v;
}
inline uint32_t le32(const uint8_t *p) {
  return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}
inline uint64_t xround(uint64_t acc, uint64_t lane) { return rotl(acc + lane * kP2, 31) * kP1; }
inline uint64_t xmerge(uint64_t h, uint64_t acc) { return (h ^ xround(0, acc)) * kP1 + kP4; }

uint64_t xxh64(const uint8_t *p, size_t len, uint64_t seed) {
  const uint8_t *end = p + len;
  uint64_t h;
  if (len >= 32) {
    uint64_t v1 = seed + kP1 + kP2, v2 = seed + kP2, v3 = seed, v4 = seed - kP1;
    for (; end - p >= 32; p += 32) {
      v1 = xround(v1, le64(p));
      v2 = xround(v2, le64(p + 8));
      v3 = xround(v3, le64(p + 16));
      v4 = xround(v4, le64(p + 24));
    }
    h = rotl(v1, 1) + rotl(v2, 7) + rotl(v3, 12) + rotl(v4, 18);
    h = xmerge(h, v1);
    h = xmerge(h, v2);
    h = xmerge(h, v3);
    h = xmerge(h, v4);
  } else {
    h = seed + kP5;
  }
  h += (uint64_t)len;
  for (; end - p >= 8; p += 8) h = rotl(h ^ xround(0, le64(p)), 27) * kP1 + kP4;
  if (end - p >= 4) {
    h = rotl(h ^ ((uint64_t)le32(p) * kP1), 23) * kP2 + kP3;
    p += 4;
  }
  for (; p < end; ++p) h = rotl(h ^ ((uint64_t)*p * kP5), 11) * kP1;
  h ^= h >> 33;
  h *= kP2;
  h ^= h >> 29;
  h *= kP3;
  h ^= h >> 32;
  return h;
}

// hash of one full block, chained on the previous block's hash
uint64_t block_hash(bool has_prefix, uint64_t prefix, const int32_t *tokens, int n) {
  std::vector<uint8_t> buf((has_prefix ? 8 : 0) + 4 * (size_t)n);
  size_t o = 0;
  if (has_prefix)
    for (int i = 0; i < 8; ++i) buf[o++] = (uint8_t)(prefix >> (8 * i));
  for (int t = 0; t < n; ++t) {
    const uint32_t v = (uint32_t)tokens[t];
    for (int i = 0; i < 4; ++i) buf[o++] = (uint8_t)(v >> (8 * i));
  }
  return xxh64(buf.data(), buf.size(), 0);
}

struct Block {
  int32_t ref = 0;
  bool hashed = false;
  uint64_t hash = 0;
  std::vector<int32_t> tokens;  // the block's token ids once it is hashed
};

}  // namespace

struct pkv_block_manager {
  int32_t block_size;
  std::vector<Block> blocks;
  std::deque<int32_t> free_list;
  std::vector<uint8_t> is_free;
  std::unordered_map<uint64_t, int32_t> by_hash;

  int32_t take_free() {  // the oldest free block, its cached identity dropped
    const int32_t b = free_list.front();
    free_list.pop_front();
    is_free[b] = 0;
    Block &bl = blocks[b];
    if (bl.hashed) {
      auto it = by_hash.find(bl.hash);
      if (it != by_hash.end() && it->second == b) by_hash.erase(it);
    }
    bl.ref = 1;
    bl.hashed = false;
    bl.hash = 0;
    bl.tokens.clear();
    return b;
  }
  void take_specific(int32_t b) {  // a cached free block that was hit: out of the free list
    for (auto it = free_list.begin(); it != free_list.end(); ++it)
      if (*it == b) {
        free_list.erase(it);
        break;
      }
    is_free[b] = 0;
    blocks[b].ref = 1;
  }
  void register_full(int32_t b, bool has_prefix, uint64_t prefix, const int32_t *tokens) {
    Block &bl = blocks[b];
    bl.hash = block_hash(has_prefix, prefix, tokens, block_size);
    bl.hashed = true;
    bl.tokens.assign(tokens, tokens + block_size);
    by_hash[bl.hash] = b;
  }
};

extern "C" {

uint64_t pkv_xxh64(const void *data, size_t len, uint64_t seed) {
  return xxh64(static_cast<const uint8_t *>(data), data ? len : 0, seed);
}

pkv_block_manager *pkv_bm_create(int32_t num_blocks, int32_t block_size) {
  if (num_blocks <= 0 || block_size <= 0) return nullptr;
  pkv_block_manager *bm = new (std::nothrow) pkv_block_manager();
  if (!bm) return nullptr;
  try {
    bm->block_size = block_size;
    bm->blocks.resize((size_t)num_blocks);
    bm->is_free.assign((size_t)num_blocks, 1);
    for (int32_t b = 0; b < num_blocks; ++b) bm->free_list.push_back(b);
  } catch (...) {
    delete bm;
    return nullptr;
  }
  return bm;
}

void pkv_bm_destroy(pkv_block_manager *bm) { delete bm; }

int32_t pkv_bm_num_free(const pkv_block_manager *bm) {
  return bm ? (int32_t)bm->free_list.size() : -1;
}

int32_t pkv_bm_ref_count(const pkv_block_manager *bm, int32_t block) {
  if (!bm || block < 0 || block >= (int32_t)bm->blocks.size()) return -1;
  return bm->blocks[(size_t)block].ref;
}

pkv_status pkv_bm_block_hash(const pkv_block_manager *bm, int32_t block, uint64_t *hash,
                             int32_t *is_hashed) {
  if (!bm || !hash || !is_hashed || block < 0 || block >= (int32_t)bm->blocks.size())
    return PKV_ERR_INVALID_ARG;
  const Block &bl = bm->blocks[(size_t)block];
  *hash = bl.hash;
  *is_hashed = bl.hashed ? 1 : 0;
  return PKV_OK;
}

pkv_status pkv_bm_allocate(pkv_block_manager *bm, const int32_t *token_ids, int32_t num_tokens,
                           int32_t *block_table, int32_t table_capacity,
                           int32_t *num_table_blocks, int32_t *num_cached_tokens) {
  if (!bm || num_tokens < 0 || (num_tokens > 0 && !token_ids) || !num_table_blocks ||
      !num_cached_tokens)
    return PKV_ERR_INVALID_ARG;
  const int32_t bs = bm->block_size;
  const int32_t nblk = (int32_t)(((int64_t)num_tokens + bs - 1) / bs);
  if (nblk > 0 && (!block_table || table_capacity < nblk)) return PKV_ERR_INVALID_ARG;
  if ((int32_t)bm->free_list.size() < nblk) return PKV_ERR_NO_BLOCKS;
  try {
    bool miss = false, has_prefix = false;
    uint64_t prefix = 0;
    int32_t cached = 0;
    for (int32_t i = 0; i < nblk; ++i) {
      const int32_t *toks = token_ids + (int64_t)i * bs;
      const int32_t n = (int32_t)((int64_t)num_tokens - (int64_t)i * bs < bs
                                      ? num_tokens - (int64_t)i * bs
                                      : bs);
      const bool full = n == bs;
      uint64_t h = 0;
      int32_t hit = -1;
      if (full && !miss) {
        h = block_hash(has_prefix, prefix, toks, bs);
        auto it = bm->by_hash.find(h);
        if (it != bm->by_hash.end() &&
            memcmp(bm->blocks[(size_t)it->second].tokens.data(), toks,
                   sizeof(int32_t) * (size_t)bs) == 0)
          hit = it->second;
      }
      int32_t b;
      if (hit < 0) {
        miss = true;
        b = bm->take_free();
        if (full) bm->register_full(b, has_prefix, prefix, toks);
      } else {
        b = hit;
        cached += bs;
        if (bm->is_free[(size_t)b]) bm->take_specific(b);
        else ++bm->blocks[(size_t)b].ref;
      }
      if (full) {
        prefix = bm->blocks[(size_t)b].hash;
        has_prefix = true;
      }
      block_table[i] = b;
    }
    *num_table_blocks = nblk;
    *num_cached_tokens = cached;
  } catch (...) {
    return PKV_ERR_INVALID_ARG;
  }
  return PKV_OK;
}

pkv_status pkv_bm_deallocate(pkv_block_manager *bm, const int32_t *block_table,
                             int32_t num_table_blocks) {
  if (!bm || num_table_blocks < 0 || (num_table_blocks > 0 && !block_table))
    return PKV_ERR_INVALID_ARG;
  // check first, so that a bad table changes nothing
  std::unordered_map<int32_t, int32_t> uses;
  for (int32_t i = 0; i < num_table_blocks; ++i) {
    const int32_t b = block_table[i];
    if (b < 0 || b >= (int32_t)bm->blocks.size()) return PKV_ERR_INVALID_ARG;
    if (++uses[b] > bm->blocks[(size_t)b].ref) return PKV_ERR_INVALID_ARG;
  }
  for (int32_t i = num_table_blocks - 1; i >= 0; --i) {  // last block first
    const int32_t b = block_table[i];
    if (--bm->blocks[(size_t)b].ref == 0) {
      bm->free_list.push_back(b);
      bm->is_free[(size_t)b] = 1;
    }
  }
  return PKV_OK;
}

int32_t pkv_bm_can_append(const pkv_block_manager *bm, int32_t seq_len) {
  if (!bm || seq_len <= 0) return 0;
  const bool needs_block = (seq_len - 1) % bm->block_size == 0;
  return (!needs_block || !bm->free_list.empty()) ? 1 : 0;
}

pkv_status pkv_bm_may_append(pkv_block_manager *bm, const int32_t *token_ids, int32_t seq_len,
                             int32_t *block_table, int32_t table_capacity,
                             int32_t *num_table_blocks) {
  if (!bm || seq_len <= 0 || !token_ids || !block_table || !num_table_blocks)
    return PKV_ERR_INVALID_ARG;
  const int32_t bs = bm->block_size;
  int32_t nb = *num_table_blocks;
  const int32_t need = (int32_t)(((int64_t)seq_len + bs - 1) / bs);
  if ((seq_len - 1) % bs == 0) {  // the new token starts a block
    if (nb != need - 1 || table_capacity < need) return PKV_ERR_INVALID_ARG;
    if (bm->free_list.empty()) return PKV_ERR_NO_BLOCKS;
    block_table[nb++] = bm->take_free();
  } else if (nb != need) {
    return PKV_ERR_INVALID_ARG;
  }
  if (seq_len % bs == 0) {  // the new token fills the last block: hash and register it
    const int32_t last = nb - 1;
    const int32_t b = block_table[last];
    if (b < 0 || b >= (int32_t)bm->blocks.size()) return PKV_ERR_INVALID_ARG;
    bool has_prefix = false;
    uint64_t prefix = 0;
    if (last > 0) {
      const Block &prev = bm->blocks[(size_t)block_table[last - 1]];
      if (!prev.hashed) return PKV_ERR_INVALID_ARG;
      has_prefix = true;
      prefix = prev.hash;
    }
    try {
      bm->register_full(b, has_prefix, prefix, token_ids + (int64_t)last * bs);
    } catch (...) {
      return PKV_ERR_INVALID_ARG;
    }
  }
  *num_table_blocks = nb;
  return PKV_OK;
}

}  // extern "C"
