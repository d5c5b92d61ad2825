"""Seeded synthetic inputs for the paged KV cache kernels and for the oracle.

This module draws numbers and lays them out; it holds none of the attention
arithmetic. Both sides of every parity check (the CUDA library and the CPU
oracle) take their inputs from here and from nowhere else.

What it produces, following the nano-vLLM pages:

* lengths: context lengths for decode, prompt lengths for prefill;
* physical block ids, handed out by a small host block allocator with a free
  list and reference counts (the block manager of «nano-vLLM 最小化vLLM重新实现»,
  架构 3 块管理器: fixed-size blocks taken from a pool, ``ref_count`` for shared
  prefix blocks);
* ``block_tables`` (per sequence, the physical block of each logical block, in
  logical order, padded with -1) and ``slot_mapping`` (per stored token, the
  flat slot ``block_id * block_size + offset`` it goes to);
* bf16 values drawn from N(0, 1), as raw ``uint16`` bit patterns.

Values for small cases come from numpy ``PCG64``; values for full-size
workloads are drawn on the device by ``device_bf16_normal`` (torch's seeded
Philox generator) because tens of GB cannot be drawn on the host in time.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 256          # tokens per KV block (nano-vLLM default)
NUM_Q_HEADS = 16          # Qwen3-0.6B attention shape
NUM_KV_HEADS = 8
HEAD_DIM = 128
NUM_LAYERS = 28
BF16_NAN_CANARY = 0x7FC1  # quiet NaN: any read of a slot nobody wrote poisons the result


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return the bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def host_bf16_normal(g: np.random.Generator, shape) -> np.ndarray:
    return f32_to_bf16_bits(g.standard_normal(shape, dtype=np.float32))


def device_bf16_normal(shape, seed: int, device="cuda"):
    """Full-size inputs: bf16 N(0,1) drawn on the device with a seeded torch generator."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    t = torch.empty(shape, dtype=torch.bfloat16, device=device)
    t.normal_(generator=gen)
    return t


# --------------------------------------------------------------------------------------
# Host block allocator (the producer of block_tables / slot_mapping; not timed)
# --------------------------------------------------------------------------------------
class BlockAllocator:
    """Free list of physical block ids in a seeded random order, with reference counts.

    ``allocate(n)`` pops the next ``n`` ids from the free list (so the first ``n`` ids of a
    seeded permutation, i.e. a uniform draw without replacement); ``share(ids)`` adds a
    reference to blocks that another sequence reuses (prefix caching); ``free(ids)`` drops a
    reference and returns blocks whose count reaches zero to the free list.
    """

    def __init__(self, num_blocks: int, g: np.random.Generator):
        self.num_blocks = int(num_blocks)
        self._free = [int(x) for x in g.permutation(self.num_blocks)]
        self._next = 0
        self.ref_count = np.zeros(self.num_blocks, dtype=np.int32)

    def allocate(self, n: int) -> list[int]:
        if self._next + n > len(self._free):
            raise MemoryError(f"pool exhausted: want {n} blocks, {len(self._free) - self._next} free")
        ids = self._free[self._next:self._next + n]
        self._next += n
        for b in ids:
            self.ref_count[b] += 1
        return ids

    def share(self, ids) -> list[int]:
        for b in ids:
            assert self.ref_count[b] > 0, "sharing a block that is not allocated"
            self.ref_count[b] += 1
        return list(ids)

    def free(self, ids) -> None:
        for b in ids:
            assert self.ref_count[b] > 0
            self.ref_count[b] -= 1
            if self.ref_count[b] == 0:
                self._free.append(int(b))


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def _pad_tables(tables: list[list[int]], width: int | None = None) -> np.ndarray:
    w = max([len(t) for t in tables] + [1]) if width is None else width
    out = np.full((len(tables), w), -1, dtype=np.int32)
    for i, t in enumerate(tables):
        out[i, :len(t)] = t
    return out


def _fill_blocks(pool: np.ndarray, table, rows: np.ndarray, block_size: int) -> None:
    """Write logical rows 0..len(rows)-1 of one sequence into its physical blocks."""
    for j in range(_cdiv(len(rows), block_size)):
        part = rows[j * block_size:(j + 1) * block_size]
        pool[int(table[j]), :len(part)] = part


def _slots(table: list[int], positions: np.ndarray, block_size: int) -> np.ndarray:
    pos = np.asarray(positions, dtype=np.int64)
    blk = np.asarray(table, dtype=np.int64)[pos // block_size]
    return blk * block_size + pos % block_size


# --------------------------------------------------------------------------------------
# Decode workloads
# --------------------------------------------------------------------------------------
@dataclass
class DecodeLayout:
    context_lens: np.ndarray            # int32 [B]; includes the token stored this step
    block_tables: np.ndarray            # int32 [B, W]; -1 padded
    slot_mapping: np.ndarray            # int64 [B]; slot of the new token (position ctx-1)
    num_blocks: int
    ref_count: np.ndarray               # int32 [num_blocks]
    block_size: int = BLOCK_SIZE
    num_q_heads: int = NUM_Q_HEADS
    num_kv_heads: int = NUM_KV_HEADS
    head_dim: int = HEAD_DIM

    @property
    def batch(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.head_dim))

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.batch else 0


def decode_layout(context_lens, num_blocks: int, g: np.random.Generator, *,
                  block_size: int = BLOCK_SIZE, num_q_heads: int = NUM_Q_HEADS,
                  num_kv_heads: int = NUM_KV_HEADS, head_dim: int = HEAD_DIM,
                  table_width: int | None = None) -> DecodeLayout:
    ctx = np.asarray(context_lens, dtype=np.int32)
    alloc = BlockAllocator(num_blocks, g)
    tables = [alloc.allocate(_cdiv(int(c), block_size)) for c in ctx]
    slots = np.array([_slots(t, [int(c) - 1], block_size)[0] if c > 0 else -1
                      for t, c in zip(tables, ctx)], dtype=np.int64)
    return DecodeLayout(ctx, _pad_tables(tables, table_width), slots, int(num_blocks),
                        alloc.ref_count, block_size, num_q_heads, num_kv_heads, head_dim)


@dataclass
class DecodeValues:
    q: np.ndarray                       # uint16 [B, Hq, D]
    k_new: np.ndarray                   # uint16 [B, Hkv, D]
    v_new: np.ndarray
    k_cache: np.ndarray                 # uint16 [NB, bs, Hkv, D]; positions < ctx-1 filled
    v_cache: np.ndarray
    logical_k: list = field(default_factory=list)   # per seq uint16 [ctx, Hkv, D]
    logical_v: list = field(default_factory=list)


def decode_values(lay: DecodeLayout, g: np.random.Generator) -> DecodeValues:
    """Draw q, the new token's k/v and the history; pre-fill the pool with the history.

    Positions 0..ctx-2 of every sequence are written to the pool here (they were stored by
    earlier steps); position ctx-1 is the new token, left for ``kv_store``. Every other slot
    holds a NaN canary.
    """
    B, Hq, Hkv, D, bs = lay.batch, lay.num_q_heads, lay.num_kv_heads, lay.head_dim, lay.block_size
    q = host_bf16_normal(g, (B, Hq, D))
    kc = np.full((lay.num_blocks, bs, Hkv, D), BF16_NAN_CANARY, dtype=np.uint16)
    vc = np.full_like(kc, BF16_NAN_CANARY)
    lk, lv = [], []
    for b in range(B):
        L = int(lay.context_lens[b])
        kb = host_bf16_normal(g, (L, Hkv, D))
        vb = host_bf16_normal(g, (L, Hkv, D))
        lk.append(kb)
        lv.append(vb)
        _fill_blocks(kc, lay.block_tables[b], kb[:max(L - 1, 0)], bs)
        _fill_blocks(vc, lay.block_tables[b], vb[:max(L - 1, 0)], bs)
    k_new = np.stack([lk[b][-1] if lay.context_lens[b] > 0 else np.zeros((Hkv, D), np.uint16)
                      for b in range(B)]) if B else np.zeros((0, Hkv, D), np.uint16)
    v_new = np.stack([lv[b][-1] if lay.context_lens[b] > 0 else np.zeros((Hkv, D), np.uint16)
                      for b in range(B)]) if B else np.zeros((0, Hkv, D), np.uint16)
    return DecodeValues(q, k_new, v_new, kc, vc, lk, lv)


def decode_values_keyed(lay: DecodeLayout, seq_ids, base_seed: int) -> DecodeValues:
    """Like decode_values, but sequence i's numbers come from their own generator seeded with
    base_seed + seq_ids[i], so a sequence draws the same values whichever shard holds it."""
    B, Hq, Hkv, D, bs = lay.batch, lay.num_q_heads, lay.num_kv_heads, lay.head_dim, lay.block_size
    kc = np.full((lay.num_blocks, bs, Hkv, D), BF16_NAN_CANARY, dtype=np.uint16)
    vc = np.full_like(kc, BF16_NAN_CANARY)
    q, lk, lv = [], [], []
    for b in range(B):
        g = rng(base_seed + int(seq_ids[b]))
        L = int(lay.context_lens[b])
        q.append(host_bf16_normal(g, (Hq, D)))
        lk.append(host_bf16_normal(g, (L, Hkv, D)))
        lv.append(host_bf16_normal(g, (L, Hkv, D)))
        _fill_blocks(kc, lay.block_tables[b], lk[-1][:max(L - 1, 0)], bs)
        _fill_blocks(vc, lay.block_tables[b], lv[-1][:max(L - 1, 0)], bs)
    return DecodeValues(np.stack(q), np.stack([x[-1] for x in lk]), np.stack([x[-1] for x in lv]),
                        kc, vc, lk, lv)


def tiny_decode(seed: int = 1):
    """Tiny decode step: 4 sequences, contexts {1, 17, 255, 300}, a pool of 8 blocks handed
    out in a seeded random permutation (1, 1, 1 and 2 blocks)."""
    g = rng(seed)
    lay = decode_layout([1, 17, 255, 300], 8, g)
    return lay, decode_values(lay, g)


def qwen3_decode_lengths(seed: int = 2, batch: int = 256, lo: int = 100, hi: int = 2048,
                         rank: int = 0, world: int = 1):
    """Qwen3-0.6B-shaped decode batch: context lengths uniform in [lo, hi]."""
    ctx = rng(seed).integers(lo, hi + 1, size=batch * world).astype(np.int32)
    return ctx[rank * batch:(rank + 1) * batch]


def qwen3_decode_layout(num_blocks: int, seed: int = 2, batch: int = 256, rank: int = 0,
                        world: int = 1) -> DecodeLayout:
    """The decode batch of one GPU. With world > 1 the global batch is batch * world
    sequences and GPU `rank` holds sequences [rank * batch, (rank + 1) * batch) in its own pool
    (sequences are independent, so the units shard with no exchange)."""
    g = rng(seed)
    ctx = g.integers(100, 2048 + 1, size=batch * world).astype(np.int32)
    return decode_layout(ctx[rank * batch:(rank + 1) * batch], num_blocks, g)


def shard_range(units: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous share [lo, hi) of `units` independent work units for one rank."""
    per, extra = divmod(units, world)
    lo = rank * per + min(rank, extra)
    return lo, lo + per + (1 if rank < extra else 0)


def long_decode_layout(num_blocks: int, seed: int = 5, batch: int = 32, ctx: int = 32768):
    return decode_layout(np.full(batch, ctx, np.int32), num_blocks, rng(seed))


def sweep_decode_layout(batch: int, num_blocks: int, seed: int = 5, ctx: int = 1024):
    return decode_layout(np.full(batch, ctx, np.int32), num_blocks, rng(seed * 1000 + batch))


def blocks_needed(context_lens, block_size: int = BLOCK_SIZE) -> int:
    return int(sum(_cdiv(int(c), block_size) for c in context_lens))


# --------------------------------------------------------------------------------------
# Prefill workloads
# --------------------------------------------------------------------------------------
@dataclass
class PrefillLayout:
    seqlens_q: np.ndarray               # int32 [N]
    seqlens_k: np.ndarray               # int32 [N]
    block_table: np.ndarray             # int32 [N, W]; -1 padded
    slot_mapping: np.ndarray            # int64 [sum seqlens_q]; slots of the query tokens' K/V
    num_blocks: int
    ref_count: np.ndarray
    prefix_len: int = 0                 # tokens of the shared prefix (prefix-cache case)
    block_size: int = BLOCK_SIZE
    num_q_heads: int = NUM_Q_HEADS
    num_kv_heads: int = NUM_KV_HEADS
    head_dim: int = HEAD_DIM

    @property
    def cu_seqlens_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.seqlens_q)]).astype(np.int32)

    @property
    def cu_seqlens_k(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.seqlens_k)]).astype(np.int32)

    @property
    def n(self) -> int:
        return int(self.seqlens_q.shape[0])

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.head_dim))


def prefill_layout(prompt_lens, num_blocks: int, g: np.random.Generator, *,
                   block_size: int = BLOCK_SIZE) -> PrefillLayout:
    """Fresh prompts: every token is a query and a key; each prompt gets private blocks."""
    L = np.asarray(prompt_lens, dtype=np.int32)
    alloc = BlockAllocator(num_blocks, g)
    tables = [alloc.allocate(_cdiv(int(x), block_size)) for x in L]
    slots = np.concatenate([_slots(t, np.arange(int(x)), block_size) for t, x in zip(tables, L)]
                           + [np.zeros(0, np.int64)]).astype(np.int64)
    return PrefillLayout(L.copy(), L.copy(), _pad_tables(tables), slots, int(num_blocks),
                         alloc.ref_count, 0, block_size)


def prefix_prefill_layout(suffix_lens, prefix_len: int, num_blocks: int, g: np.random.Generator,
                          *, block_size: int = BLOCK_SIZE, private_prefix: bool = False
                          ) -> PrefillLayout:
    """Sequences that share one cached prefix of ``prefix_len`` tokens (a whole number of
    blocks, held once with ref_count = number of users) plus a private suffix. Queries are the
    suffix tokens only; keys are prefix + suffix, read through ``block_table``.

    With ``private_prefix`` every sequence gets its own copy of the prefix blocks instead
    (same contents, other physical ids) -- the "private copy" side of the sharing invariant.
    """
    assert prefix_len % block_size == 0
    S = np.asarray(suffix_lens, dtype=np.int32)
    alloc = BlockAllocator(num_blocks, g)
    npre = prefix_len // block_size
    shared = alloc.allocate(npre)          # the first sequence computes and owns the prefix
    tables, slots = [], []
    for i, s in enumerate(S):
        if i == 0:
            pre = shared
        else:
            pre = alloc.allocate(npre) if private_prefix else alloc.share(shared)
        own = alloc.allocate(_cdiv(int(s), block_size))
        t = list(pre) + list(own)
        tables.append(t)
        slots.append(_slots(t, prefix_len + np.arange(int(s)), block_size))
    slots = np.concatenate(slots + [np.zeros(0, np.int64)]).astype(np.int64)
    return PrefillLayout(S.copy(), (S + prefix_len).astype(np.int32), _pad_tables(tables), slots,
                         int(num_blocks), alloc.ref_count, prefix_len, block_size)


def varlen_prefill_lengths(seed: int = 3, n: int = 256, lo: int = 100, hi: int = 1024):
    """Varlen causal prefill: prompt lengths uniform in [lo, hi]."""
    return rng(seed).integers(lo, hi + 1, size=n).astype(np.int32)


def varlen_prefill_layout(num_blocks: int, seed: int = 3, n: int = 256) -> PrefillLayout:
    g = rng(seed)
    L = g.integers(100, 1024 + 1, size=n).astype(np.int32)
    return prefill_layout(L, num_blocks, g)


def prefix_prefill_case_layout(num_blocks: int, seed: int = 4, n: int = 64,
                               prefix_len: int = 2048) -> PrefillLayout:
    """Prefix-cached prefill: n sequences share one 2048-token prefix (8 shared blocks), each
    with a suffix of uniform length in [256, 768]."""
    g = rng(seed)
    S = g.integers(256, 768 + 1, size=n).astype(np.int32)
    return prefix_prefill_layout(S, prefix_len, num_blocks, g)


@dataclass
class PrefillValues:
    q: np.ndarray                       # uint16 [Tq, Hq, D]
    k: np.ndarray                       # uint16 [Tk, Hkv, D]  packed keys (all of every sequence)
    v: np.ndarray
    k_cache: np.ndarray                 # uint16 [NB, bs, Hkv, D]; shared prefix pre-filled
    v_cache: np.ndarray


def prefill_values(lay: PrefillLayout, g: np.random.Generator) -> PrefillValues:
    """Queries for the new tokens; keys/values for every key position. For prefix-cache
    layouts the prefix part of each sequence's keys is one shared draw, pre-filled into the
    shared blocks; the suffix tokens' K/V are left for ``kv_store``."""
    Hq, Hkv, D, bs = lay.num_q_heads, lay.num_kv_heads, lay.head_dim, lay.block_size
    Tq = int(lay.seqlens_q.sum())
    q = host_bf16_normal(g, (Tq, Hq, D))
    kc = np.full((lay.num_blocks, bs, Hkv, D), BF16_NAN_CANARY, dtype=np.uint16)
    vc = np.full_like(kc, BF16_NAN_CANARY)
    P = lay.prefix_len
    pk = host_bf16_normal(g, (P, Hkv, D))
    pv = host_bf16_normal(g, (P, Hkv, D))
    ks, vs = [], []
    for n in range(lay.n):
        s = int(lay.seqlens_q[n])
        sk = host_bf16_normal(g, (s, Hkv, D))
        sv = host_bf16_normal(g, (s, Hkv, D))
        ks.append(np.concatenate([pk, sk]))
        vs.append(np.concatenate([pv, sv]))
        _fill_blocks(kc, lay.block_table[n], pk, bs)
        _fill_blocks(vc, lay.block_table[n], pv, bs)
    k = np.concatenate(ks + [np.zeros((0, Hkv, D), np.uint16)])
    v = np.concatenate(vs + [np.zeros((0, Hkv, D), np.uint16)])
    return PrefillValues(q, k, v, kc, vc)


def suffix_rows(lay: PrefillLayout) -> np.ndarray:
    """Row indices, into the packed keys, of the tokens that are queries (the suffixes)."""
    cu_k = lay.cu_seqlens_k
    return np.concatenate([cu_k[n] + lay.prefix_len + np.arange(int(lay.seqlens_q[n]))
                           for n in range(lay.n)] + [np.zeros(0, np.int64)]).astype(np.int64)


def random_cos_sin_table(g: np.random.Generator, max_position: int, head_dim: int) -> np.ndarray:
    """[max_position, head_dim] float32: cosines of seeded random angles in [-pi, pi), then
    their sines -- an arbitrary rotation table of the layout the RoPE step reads (the
    kernels and the oracle take any table; none of the method is in how it is drawn)."""
    a = g.uniform(-np.pi, np.pi, (max_position, head_dim // 2))
    return np.concatenate([np.cos(a), np.sin(a)], axis=1).astype(np.float32)
