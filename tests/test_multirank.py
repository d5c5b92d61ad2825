"""The multi-GPU path on CPU: world_size 2 over gloo.

Decode units (sequences) are independent, so N GPUs each take their own contiguous share of
a global batch, in their own pool, with no data exchange; only the benchmark's timing takes
a max over ranks. Here each rank runs the oracle (store + paged decode) on its share; the
gathered shares must equal one process running the whole batch, bit for bit, and the timing
reduction must return the slowest rank's time.
"""
import os
import socket
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GLOBAL_BATCH, SEED = 10, 9


def _run_shard(rank, world):
    import oracle
    import workloads as w
    g = w.rng(SEED)
    ctx_all = g.integers(1, 700, size=GLOBAL_BATCH).astype(np.int32)
    lo, hi = w.shard_range(GLOBAL_BATCH, rank, world)
    ctx = ctx_all[lo:hi]
    lay = w.decode_layout(ctx, w.blocks_needed(ctx) + 3, w.rng(100 + rank + 10 * world),
                          num_q_heads=4, num_kv_heads=2, table_width=3)
    val = w.decode_values_keyed(lay, np.arange(lo, hi), 5000)
    kc, vc = val.k_cache.copy(), val.v_cache.copy()
    oracle.kv_store(val.k_new, val.v_new, lay.slot_mapping, kc, vc)
    return oracle.paged_decode(val.q, kc, vc, lay.block_tables, lay.context_lens, lay.scale)


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        out = torch.from_numpy(_run_shard(rank, world))
        sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(sizes, torch.tensor([out.shape[0]]))
        pad = torch.zeros((int(max(s.item() for s in sizes)),) + tuple(out.shape[1:]),
                          dtype=out.dtype)
        pad[:out.shape[0]] = out
        got = [torch.zeros_like(pad) for _ in range(world)]
        dist.all_gather(got, pad)                      # test-only: collect the shards
        slowest = bench.max_over_ranks(1.0 + rank, world)
        if rank == 0:
            full = torch.cat([t[:int(s.item())] for t, s in zip(got, sizes)]).numpy()
            q.put((full, slowest))
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_ranks_shard_sequences_with_identical_results():
    sys.path.insert(0, ROOT)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    full, slowest = q.get(timeout=240)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    single = _run_shard(0, 1)
    assert full.shape == single.shape
    assert np.array_equal(full, single)
    assert slowest == 2.0


def test_shard_ranges_cover_every_unit_once():
    import workloads as w
    for units in (0, 1, 7, 256, 257):
        for world in (1, 2, 3, 8):
            spans = [w.shard_range(units, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == units
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            assert max(h - l for l, h in spans) - min(h - l for l, h in spans) <= 1
