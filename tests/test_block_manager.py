"""Host block manager: the oracle pinned to published values and to the invariants the pages'
design implies, then the library's C++ manager (pkv_bm_*) checked against the oracle step by
step on random workloads (allocate with shared prefixes, decode appends, preemption, finish).
CPU only: the block manager is host code.
"""
import random

import pytest

import paged_kv_cache_208_gb300 as pkv
from oracle.block_manager import BlockManagerOracle, NoBlocks, block_hash, xxh64

import block_manager_pins as pins
from block_manager_pins import XXH64_VECTORS

bm_oracle = __import__("oracle.block_manager", fromlist=["*"])


# ------------------------------------------------------------------------------ oracle pins
@pytest.mark.parametrize("data,want", XXH64_VECTORS)
def test_oracle_xxh64_published_values(data, want):
    assert xxh64(data) == want


@pytest.mark.parametrize("pin", pins.ALL_PINS[1:], ids=[f.__name__ for f in pins.ALL_PINS[1:]])
def test_oracle_pin(pin):
    pin(bm_oracle)


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
