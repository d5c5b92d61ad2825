"""Block manager oracle -- TEST INFRASTRUCTURE ONLY.

A plain, slow restatement of the host block manager that the library implements in C++ (the
`pkv_bm_*` calls), used by `tests/` to check the library's behaviour step by step. Nothing in
the product path imports this module.

What it follows: «nano-vLLM 最小化vLLM重新实现», 架构 3 (块管理器) -- a pool of fixed-size
blocks, each with a reference count and a hash; allocate() reuses cached blocks whose hash
matches and takes new blocks only for the rest of the sequence; block hashes are xxhash over
the token ids; preemption frees a sequence's blocks -- with the per-sequence block list as the
page table of «企业官网建设流程全解析 (Nano-vLLM 指南)» §2.2 and prefix reuse as its §4.4.
The pages give the idea, not the rules; the readings taken here (also stated in the C++):

  * only full blocks are hashed; hash = XXH64(seed 0) of the previous block's hash as 8
    little-endian bytes (nothing for a sequence's first block) followed by the token ids as
    4-byte little-endian integers; a hit also needs equal token ids;
  * after the first miss of a sequence, the rest of it gets new blocks;
  * free blocks are handed out first-in first-out (0, 1, 2, ... at the start); a freed block
    keeps its hash and stays a possible hit until it is handed out again;
  * allocating needs as many free blocks as the sequence has blocks, else nothing changes;
  * after appending a token to a sequence of now n tokens: a new block when position n - 1
    starts a block, and the last block is hashed when n fills it.

XXH64 below is written from the published xxHash specification (64-bit variant): four
accumulators over 32-byte stripes, a merge, then 8-, 4- and 1-byte tail steps and a final
avalanche.
"""
from __future__ import annotations

M64 = (1 << 64) - 1
P1, P2, P3, P4, P5 = (0x9E3779B185EBCA87, 0xC2B2AE3D27D4EB4F, 0x165667B19E3779F9,
                      0x85EBCA77C2B2AE63, 0x27D4EB2F165667C5)


def _rotl(x: int, r: int) -> int:
    return ((x << r) | (x >> (64 - r))) & M64


def _round(acc: int, lane: int) -> int:
    acc = (acc + lane * P2) & M64
    return (_rotl(acc, 31) * P1) & M64


def xxh64(data: bytes, seed: int = 0) -> int:
    n = len(data)
    i = 0
    if n >= 32:
        v = [(seed + P1 + P2) & M64, (seed + P2) & M64, seed & M64, (seed - P1) & M64]
        while n - i >= 32:
            for j in range(4):
                v[j] = _round(v[j], int.from_bytes(data[i + 8 * j:i + 8 * j + 8], "little"))
            i += 32
        h = (_rotl(v[0], 1) + _rotl(v[1], 7) + _rotl(v[2], 12) + _rotl(v[3], 18)) & M64
        for j in range(4):
            h = ((h ^ _round(0, v[j])) * P1 + P4) & M64
    else:
        h = (seed + P5) & M64
    h = (h + n) & M64
    while n - i >= 8:
        h ^= _round(0, int.from_bytes(data[i:i + 8], "little"))
        h = (_rotl(h, 27) * P1 + P4) & M64
        i += 8
    if n - i >= 4:
        h ^= (int.from_bytes(data[i:i + 4], "little") * P1) & M64
        h = (_rotl(h, 23) * P2 + P3) & M64
        i += 4
    while i < n:
        h ^= (data[i] * P5) & M64
        h = (_rotl(h, 11) * P1) & M64
        i += 1
    h ^= h >> 33
    h = (h * P2) & M64
    h ^= h >> 29
    h = (h * P3) & M64
    h ^= h >> 32
    return h


def block_hash(prefix, tokens) -> int:
    """Hash of one full block; prefix = the previous block's hash, or None for the first."""
    data = b"" if prefix is None else prefix.to_bytes(8, "little")
    data += b"".join((t & 0xFFFFFFFF).to_bytes(4, "little") for t in tokens)
    return xxh64(data, 0)


class NoBlocks(Exception):
    pass


class BlockManagerOracle:
    def __init__(self, num_blocks: int, block_size: int):
        self.bs = block_size
        self.ref = [0] * num_blocks
        self.hash = [None] * num_blocks        # None until the block is full and registered
        self.tokens = [None] * num_blocks
        self.free = list(range(num_blocks))     # front = next to hand out
        self.table_of_hash = {}

    def num_free(self) -> int:
        return len(self.free)

    def _take_free(self) -> int:
        b = self.free.pop(0)
        if self.hash[b] is not None and self.table_of_hash.get(self.hash[b]) == b:
            del self.table_of_hash[self.hash[b]]
        self.ref[b] = 1
        self.hash[b] = None
        self.tokens[b] = None
        return b

    def _register(self, b, prefix, toks):
        self.hash[b] = block_hash(prefix, toks)
        self.tokens[b] = list(toks)
        self.table_of_hash[self.hash[b]] = b

    def allocate(self, token_ids):
        bs = self.bs
        blocks = [list(token_ids[i:i + bs]) for i in range(0, len(token_ids), bs)]
        if len(self.free) < len(blocks):
            raise NoBlocks()
        table, cached, missed, prefix = [], 0, False, None
        for toks in blocks:
            full = len(toks) == bs
            hit = None
            if full and not missed:
                h = block_hash(prefix, toks)
                b = self.table_of_hash.get(h)
                if b is not None and self.tokens[b] == toks:
                    hit = b
            if hit is None:
                missed = True
                b = self._take_free()
                if full:
                    self._register(b, prefix, toks)
            else:
                b = hit
                cached += bs
                if b in self.free:
                    self.free.remove(b)
                    self.ref[b] = 1
                else:
                    self.ref[b] += 1
            if full:
                prefix = self.hash[b]
            table.append(b)
        return table, cached

    def deallocate(self, table):
        for b in reversed(table):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)

    def can_append(self, seq_len: int) -> bool:
        return (seq_len - 1) % self.bs != 0 or len(self.free) > 0

    def may_append(self, token_ids, table):
        n, bs = len(token_ids), self.bs
        table = list(table)
        if (n - 1) % bs == 0:
            if not self.free:
                raise NoBlocks()
            table.append(self._take_free())
        if n % bs == 0:
            last = len(table) - 1
            prefix = self.hash[table[last - 1]] if last > 0 else None
            self._register(table[last], prefix, token_ids[last * bs:(last + 1) * bs])
        return table
