"""Pins of the block manager oracle (oracle/block_manager.py), written against a module
argument so that tests/test_oracle_mutants.py can run them on planted mistakes as well.

Each pin raises AssertionError when the module misbehaves: published XXH64 values, the hash
chaining, prefix hits with FIFO block hand-out, cached blocks surviving until they are handed
out again, a failed allocation changing nothing, decode appends, a forged hash collision that
must miss, and invariants over random workloads.
"""
import random

# published XXH64 (seed 0) values of short strings
XXH64_VECTORS = [
    (b"", 0xEF46DB3751D8E999),
    (b"a", 0xD24EC4F1A98C6E5B),
    (b"abc", 0x44BC2CF5AD770999),
    (b"Nobody inspects the spammish repetition", 0xFBCEA83C8A378BF1),
]


def pin_xxh64_published_values(mod):
    for data, want in XXH64_VECTORS:
        assert mod.xxh64(data) == want, data


def pin_block_hash_is_chained(mod):
    a, b = [1, 2, 3, 4], [5, 6, 7, 8]
    h0 = mod.block_hash(None, a)
    assert h0 == mod.xxh64(b"".join(t.to_bytes(4, "little") for t in a))
    assert mod.block_hash(h0, b) == mod.xxh64(h0.to_bytes(8, "little") +
                                              b"".join(t.to_bytes(4, "little") for t in b))
    # the same tokens after a different prefix hash differently
    assert mod.block_hash(mod.block_hash(None, [9, 9, 9, 9]), b) != mod.block_hash(h0, b)


def check_invariants(m, live):
    """Free list and held blocks partition the pool; reference counts equal the number of
    live tables that hold a block; every live table covers its sequence."""
    held = [b for b in range(len(m.ref)) if m.ref[b] > 0]
    assert sorted(held + m.free) == list(range(len(m.ref)))
    assert len(set(m.free)) == len(m.free)
    count = {}
    for toks, table in live.values():
        assert len(table) == -(-len(toks) // m.bs)
        for b in table:
            count[b] = count.get(b, 0) + 1
    assert count == {b: m.ref[b] for b in held}


def pin_prefix_hits_and_fifo(mod):
    m = mod.BlockManagerOracle(8, 4)
    t1, c1 = m.allocate(list(range(10)))              # two full blocks + a partial one
    assert (t1, c1) == ([0, 1, 2], 0)
    t2, c2 = m.allocate(list(range(8)) + [77, 78])    # shares the two full blocks
    assert (t2, c2) == ([0, 1, 3], 8) and m.ref[0] == m.ref[1] == 2
    t3, c3 = m.allocate([0, 1, 2, 3, 9, 9, 9, 9])     # shares the first block only
    assert (t3, c3) == ([0, 4], 4)
    t4, _ = m.allocate([5, 1, 2, 3, 4, 5, 6, 7])      # first block misses: nothing shared
    assert t4 == [5, 6]
    m.deallocate(t1)
    m.deallocate(t2)
    # freed blocks join the back of the list, each table's last block first; block 0 is
    # still held by t3
    assert m.free == [7, 2, 3, 1]
    # the freed-but-cached prefix is still a hit
    t5, c5 = m.allocate(list(range(8)))
    assert (t5, c5) == ([0, 1], 8)


def pin_cache_survives_until_reuse(mod):
    m = mod.BlockManagerOracle(4, 2)
    t, _ = m.allocate([1, 2, 3, 4])
    assert t == [0, 1]
    m.deallocate(t)                                    # free list: 2, 3, 1, 0
    assert m.allocate([1, 2, 3, 4]) == ([0, 1], 4)     # both blocks still cached
    m.deallocate([0, 1])                               # free list: 2, 3, 1, 0
    t2, _ = m.allocate([7, 7, 8, 8, 9, 9])             # hands out 2, 3, 1
    assert t2 == [2, 3, 1]
    m.deallocate(t2)                                   # free list: 0, 1, 3, 2
    # block 0 still holds [1, 2]; block 1 was handed out again, so [3, 4] misses
    assert m.allocate([1, 2, 3, 4]) == ([0, 1], 2)


def pin_no_blocks_changes_nothing(mod):
    m = mod.BlockManagerOracle(3, 4)
    m.allocate(list(range(8)))
    before = (list(m.ref), list(m.free), dict(m.table_of_hash))
    try:
        m.allocate(list(range(100, 109)))              # needs 3 blocks, 1 free
        raised = False
    except mod.NoBlocks:
        raised = True
    assert raised
    assert (list(m.ref), list(m.free), dict(m.table_of_hash)) == before


def pin_decode_appends(mod):
    m = mod.BlockManagerOracle(10, 4)
    toks = [1, 2, 3]
    table, _ = m.allocate(toks)
    for t in range(4, 14):
        toks.append(t)
        assert m.can_append(len(toks))
        table = m.may_append(toks, table)
        assert len(table) == -(-len(toks) // 4)
        full = len(toks) // 4
        assert all(m.hash[b] is not None for b in table[:full])
        if len(toks) % 4:
            assert m.hash[table[-1]] is None
    # the appended blocks are hits for a new sequence with the same tokens
    assert m.allocate(toks)[1] == 12


def pin_hit_needs_equal_tokens(mod):
    """A hash that names a block holding other tokens (a collision, forged here) is a miss."""
    m = mod.BlockManagerOracle(4, 2)
    t, _ = m.allocate([1, 2])
    m.table_of_hash[mod.block_hash(None, [3, 4])] = t[0]
    t2, c2 = m.allocate([3, 4])
    assert c2 == 0 and t2 != t


def pin_random_invariants(mod):
    rng = random.Random(7)
    for bs in (1, 2, 4):
        m = mod.BlockManagerOracle(24, bs)
        live, nxt = {}, 0
        prefixes = [[rng.randrange(5) for _ in range(rng.randrange(1, 9))] for _ in range(4)]
        for _ in range(300):
            op = rng.random()
            if op < 0.4:
                toks = rng.choice(prefixes) + [rng.randrange(5) for _ in range(rng.randrange(6))]
                if not toks:
                    continue
                try:
                    table, cached = m.allocate(toks)
                except mod.NoBlocks:
                    continue
                assert cached % bs == 0 and cached <= len(toks)
                live[nxt] = (toks, table)
                nxt += 1
            elif op < 0.75 and live:
                k = rng.choice(list(live))
                toks, table = live[k]
                toks = toks + [rng.randrange(5)]
                if m.can_append(len(toks)):
                    live[k] = (toks, m.may_append(toks, table))
            elif live:
                k = rng.choice(list(live))
                m.deallocate(live.pop(k)[1])
            check_invariants(m, live)


ALL_PINS = [pin_xxh64_published_values, pin_block_hash_is_chained, pin_prefix_hits_and_fifo,
            pin_cache_survives_until_reuse, pin_no_blocks_changes_nothing, pin_decode_appends,
            pin_hit_needs_equal_tokens, pin_random_invariants]
