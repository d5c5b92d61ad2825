"""Host block manager: the oracle pinned to published values and to the invariants the pages'
design implies, then the library's C++ manager (pkv_bm_*) checked against the oracle step by
step on random workloads (allocate with shared prefixes, decode appends, preemption, finish).
CPU only: the block manager is host code.
"""
import random

import pytest

import paged_kv_cache_208_gb300 as pkv
from oracle.block_manager import BlockManagerOracle, NoBlocks, block_hash, xxh64

# published XXH64 (seed 0) values of short strings
XXH64_VECTORS = [
    (b"", 0xEF46DB3751D8E999),
    (b"a", 0xD24EC4F1A98C6E5B),
    (b"abc", 0x44BC2CF5AD770999),
    (b"Nobody inspects the spammish repetition", 0xFBCEA83C8A378BF1),
]


# ------------------------------------------------------------------------------ oracle pins
@pytest.mark.parametrize("data,want", XXH64_VECTORS)
def test_oracle_xxh64_published_values(data, want):
    assert xxh64(data) == want


def test_oracle_block_hash_is_chained():
    a, b = [1, 2, 3, 4], [5, 6, 7, 8]
    h0 = block_hash(None, a)
    assert h0 == xxh64(b"".join(t.to_bytes(4, "little") for t in a))
    assert block_hash(h0, b) == xxh64(h0.to_bytes(8, "little") +
                                      b"".join(t.to_bytes(4, "little") for t in b))
    # the same tokens after a different prefix hash differently
    assert block_hash(block_hash(None, [9, 9, 9, 9]), b) != block_hash(h0, b)


def _invariants(m: BlockManagerOracle, live):
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


def test_oracle_prefix_hits_and_fifo():
    m = BlockManagerOracle(8, 4)
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


def test_oracle_cache_survives_until_reuse():
    m = BlockManagerOracle(4, 2)
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


def test_oracle_no_blocks_changes_nothing():
    m = BlockManagerOracle(3, 4)
    m.allocate(list(range(8)))
    before = (list(m.ref), list(m.free), dict(m.table_of_hash))
    with pytest.raises(NoBlocks):
        m.allocate(list(range(100, 109)))           # needs 3 blocks, 1 free
    assert (list(m.ref), list(m.free), dict(m.table_of_hash)) == before


def test_oracle_decode_appends():
    m = BlockManagerOracle(10, 4)
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


def test_oracle_random_invariants():
    rng = random.Random(7)
    for bs in (1, 2, 4):
        m = BlockManagerOracle(24, bs)
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
                except NoBlocks:
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
            _invariants(m, live)


# ------------------------------------------------------------------- library vs the oracle
def _same_state(lib: pkv.BlockManager, m: BlockManagerOracle):
    assert lib.num_free == m.num_free()
    for b in range(len(m.ref)):
        assert lib.ref_count(b) == m.ref[b], b
        assert lib.block_hash(b) == m.hash[b], b


@pytest.mark.parametrize("bs", [1, 2, 4, 16, 256])
def test_library_matches_oracle_on_random_workload(bs):
    rng = random.Random(100 + bs)
    nblocks = 40
    lib, m = pkv.BlockManager(nblocks, bs), BlockManagerOracle(nblocks, bs)
    vocab = 3 if bs <= 4 else 50
    prefixes = [[rng.randrange(vocab) for _ in range(rng.randrange(1, 3 * bs + 2))]
                for _ in range(5)]
    live_lib, live_or, nxt = {}, {}, 0
    for _ in range(400):
        op = rng.random()
        if op < 0.35:
            toks = rng.choice(prefixes) + [rng.randrange(vocab)
                                           for _ in range(rng.randrange(2 * bs + 1))]
            try:
                want = m.allocate(toks)
            except NoBlocks:
                with pytest.raises(pkv.PkvError) as e:
                    lib.allocate(toks)
                assert e.value.status == pkv.ERR_NO_BLOCKS
                _same_state(lib, m)
                continue
            assert lib.allocate(toks) == want
            live_or[nxt] = (toks, want[0])
            live_lib[nxt] = (toks, want[0])
            nxt += 1
        elif op < 0.8 and live_or:
            k = rng.choice(list(live_or))
            toks = live_or[k][0] + [rng.randrange(vocab)]
            assert lib.can_append(len(toks)) == m.can_append(len(toks))
            if not m.can_append(len(toks)):
                continue
            t_or = m.may_append(toks, live_or[k][1])
            t_lib = lib.may_append(toks, live_lib[k][1])
            assert t_lib == t_or
            live_or[k] = (toks, t_or)
            live_lib[k] = (toks, t_lib)
        elif live_or:
            k = rng.choice(list(live_or))
            m.deallocate(live_or.pop(k)[1])
            lib.deallocate(live_lib.pop(k)[1])
        _same_state(lib, m)


@pytest.mark.parametrize("data,want", XXH64_VECTORS)
def test_library_xxh64(data, want):
    assert pkv.xxh64(data) == want


def test_library_xxh64_matches_oracle_on_all_tail_lengths():
    rng = random.Random(3)
    for n in range(0, 100):
        data = bytes(rng.randrange(256) for _ in range(n))
        for seed in (0, 1, 2 ** 63 + 5):
            assert pkv.xxh64(data, seed) == xxh64(data, seed), (n, seed)


def test_library_errors_change_nothing():
    assert not pkv.lib().pkv_bm_create(0, 4)
    assert not pkv.lib().pkv_bm_create(4, 0)
    lib = pkv.BlockManager(4, 2)
    t, _ = lib.allocate([1, 2, 3])
    with pytest.raises(pkv.PkvError) as e:
        lib.deallocate([t[0], t[0]])                 # released more often than held
    assert e.value.status == pkv.ERR_INVALID_ARG
    with pytest.raises(pkv.PkvError):
        lib.deallocate([9])                          # out of range
    assert lib.num_free == 2 and lib.ref_count(t[0]) == 1
    with pytest.raises(pkv.PkvError) as e:
        lib.allocate(list(range(7)))                 # needs 4 blocks, 2 free
    assert e.value.status == pkv.ERR_NO_BLOCKS and lib.num_free == 2
    with pytest.raises(pkv.PkvError):
        lib.may_append(list(range(7)), t)            # the table covers 3 tokens, not 6
