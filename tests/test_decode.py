"""Paged decode attention on the GPU against the oracle, through the C ABI.

Element-wise parity within |err| <= 1e-2 + 1e-2 |ref| on every output, at small sizes that
span several tiles, splits and blocks with ragged tails, and at the full decode workloads
(Qwen3 batch of 256, 32 x 32k, the batch sweep) in the launch configuration the benchmark
times; plus the invariants: bit-identical results under block permutation and for shared
vs private prefix blocks, and a one-token context returning V exactly.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads as w
from gpu_util import (assert_attention_close, compact_for_oracle, dev, fill_sequences_on_device,
                      host_bits)
from libbuild import build_and_import

pytestmark = pytest.mark.gpu
pkv = build_and_import()


def _gpu_step(lay, kc_d, vc_d, q_d, k_new_d, v_new_d, num_splits=0, store=True):
    if store:
        pkv.kv_store(k_new_d, v_new_d, dev(lay.slot_mapping), kc_d, vc_d)
    return pkv.paged_decode_attn(q_d, kc_d, vc_d, dev(lay.block_tables), dev(lay.context_lens),
                                 lay.max_context_len, lay.scale, num_splits=num_splits)


def _host_case(ctx, nb_spare=4, seed=0, hq=16, hkv=8, table_width=None):
    g = w.rng(seed)
    lay = w.decode_layout(ctx, w.blocks_needed(ctx) + nb_spare, g, num_q_heads=hq,
                          num_kv_heads=hkv, table_width=table_width)
    return lay, w.decode_values(lay, g)


def _oracle_step(lay, val):
    kc, vc = val.k_cache.copy(), val.v_cache.copy()
    oracle.kv_store(val.k_new, val.v_new, lay.slot_mapping, kc, vc)
    return oracle.paged_decode(val.q, kc, vc, lay.block_tables, lay.context_lens, lay.scale)


@pytest.mark.parametrize("num_splits", [0, 1, 2, 3, 5])
def test_decode_tiny_step(num_splits):
    """Tiny decode step: contexts {1, 17, 255, 300}, a pool of 8 blocks in a seeded random
    permutation; store the new tokens, then attend."""
    lay, val = w.tiny_decode()
    ref = _oracle_step(lay, val)
    out = _gpu_step(lay, dev(val.k_cache), dev(val.v_cache), dev(val.q), dev(val.k_new),
                    dev(val.v_new), num_splits)
    assert_attention_close(out, ref, f"tiny splits={num_splits}")
    # context of one token: the output is that token's V, exactly
    v0 = np.repeat(val.logical_v[0][0], 2, axis=0)
    assert np.array_equal(host_bits(out)[0], v0)
    assert pkv.get_device_errors() == 0


@pytest.mark.parametrize("seed,ctx", [
    (11, [1, 2, 63, 64, 65, 127, 128, 129]),
    (12, [255, 256, 257, 511, 512, 513, 1000, 1500]),
    (13, [3000, 17, 4097, 700]),
])
@pytest.mark.parametrize("num_splits", [0, 1, 4, 8, 9])
def test_decode_ragged_contexts(seed, ctx, num_splits):
    lay, val = _host_case(ctx, seed=seed)
    ref = _oracle_step(lay, val)
    out = _gpu_step(lay, dev(val.k_cache), dev(val.v_cache), dev(val.q), dev(val.k_new),
                    dev(val.v_new), num_splits)
    assert_attention_close(out, ref, f"ctx={ctx} splits={num_splits}")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 4), (16, 2), (12, 4), (16, 16)])
def test_decode_head_groupings(hq, hkv):
    lay, val = _host_case([5, 300, 129], seed=21, hq=hq, hkv=hkv)
    ref = _oracle_step(lay, val)
    out = _gpu_step(lay, dev(val.k_cache), dev(val.v_cache), dev(val.q), dev(val.k_new),
                    dev(val.v_new))
    assert_attention_close(out, ref, f"hq={hq} hkv={hkv}")


def test_decode_block_permutation_is_bit_identical():
    lay, val = _host_case([700, 90, 1025, 256], nb_spare=9, seed=31)
    kc, vc = val.k_cache.copy(), val.v_cache.copy()
    oracle.kv_store(val.k_new, val.v_new, lay.slot_mapping, kc, vc)
    base = pkv.paged_decode_attn(dev(val.q), dev(kc), dev(vc), dev(lay.block_tables),
                                 dev(lay.context_lens), lay.max_context_len, lay.scale)
    perm = w.rng(7).permutation(lay.num_blocks)
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    bt2 = np.where(lay.block_tables >= 0, perm[np.maximum(lay.block_tables, 0)], -1)
    moved = pkv.paged_decode_attn(dev(val.q), dev(kc2), dev(vc2), dev(bt2.astype(np.int32)),
                                  dev(lay.context_lens), lay.max_context_len, lay.scale)
    assert np.array_equal(host_bits(base), host_bits(moved))


def test_decode_shared_prefix_block_equals_private_copy():
    """Sequences whose first blocks are one ref-counted shared block give the same bits as
    sequences holding private copies of that block."""
    g = w.rng(41)
    nb, bs = 16, 256
    shared_rows_k = w.host_bf16_normal(g, (bs, 8, 128))
    shared_rows_v = w.host_bf16_normal(g, (bs, 8, 128))
    ctx = np.array([300, 600, 257], np.int32)
    alloc = w.BlockAllocator(nb, g)
    pre = alloc.allocate(1)
    t_shared, t_private = [], []
    for i, c in enumerate(ctx):
        own = alloc.allocate(-(-int(c) // bs) - 1)
        t_shared.append((pre if i == 0 else alloc.share(pre)) + own)
        t_private.append(alloc.allocate(1) + own)
    kc = w.host_bf16_normal(g, (nb, bs, 8, 128))
    vc = w.host_bf16_normal(g, (nb, bs, 8, 128))
    for t in t_shared + t_private:
        kc[t[0]], vc[t[0]] = shared_rows_k, shared_rows_v
    q = w.host_bf16_normal(g, (3, 16, 128))
    outs = []
    for tabs in (t_shared, t_private):
        bt = w._pad_tables(tabs)
        outs.append(host_bits(pkv.paged_decode_attn(dev(q), dev(kc), dev(vc), dev(bt), dev(ctx),
                                                    int(ctx.max()), 128 ** -0.5)))
    assert alloc.ref_count[pre[0]] == 3
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("num_splits", [0, 1, 4, 8, 9])
def test_decode_stale_table_entries_past_context(num_splits):
    """Table entries past each context hold valid block ids of other sequences (a row left
    over from an earlier step): nothing past the context may be read. Units whose first
    tile lies past their context (the kernel may start loading them before it has read the
    context length) must drop that tile."""
    lay, val = _host_case([5, 300, 2100, 40], seed=57)  # 9 splits: 288 units, a static grid
    g = w.rng(58)
    bt = lay.block_tables.copy()
    stale = bt < 0
    bt[stale] = g.integers(0, lay.num_blocks, size=int(stale.sum()))
    ref = _oracle_step(lay, val)
    lay_stale = dataclasses.replace(lay, block_tables=bt)
    out = _gpu_step(lay_stale, dev(val.k_cache), dev(val.v_cache), dev(val.q), dev(val.k_new),
                    dev(val.v_new), num_splits)
    assert_attention_close(out, ref, f"stale table entries, splits={num_splits}")
    assert pkv.get_device_errors() == 0


def test_decode_zero_query_is_mean_of_v():
    lay, val = _host_case([400, 33], seed=51)
    kc, vc = val.k_cache.copy(), val.v_cache.copy()
    oracle.kv_store(val.k_new, val.v_new, lay.slot_mapping, kc, vc)
    q0 = np.zeros_like(val.q)
    out = pkv.paged_decode_attn(dev(q0), dev(kc), dev(vc), dev(lay.block_tables),
                                dev(lay.context_lens), lay.max_context_len, lay.scale)
    want = np.stack([np.repeat(w.bf16_bits_to_f32(val.logical_v[b]).astype(np.float64)
                               .mean(axis=0), 2, axis=0) for b in range(2)])
    assert_attention_close(out, want, "q=0")


def test_decode_empty_context_gives_zeros():
    lay, val = _host_case([5, 300], seed=61)
    ctx = lay.context_lens.copy()
    ctx[0] = 0
    for ns in (1, 0):
        out = pkv.paged_decode_attn(dev(val.q), dev(val.k_cache), dev(val.v_cache),
                                    dev(lay.block_tables), dev(ctx), 300, lay.scale,
                                    num_splits=ns)
        assert not host_bits(out)[0].any()


def test_decode_bad_block_id_is_flagged_not_faulted():
    lay, val = _host_case([300, 40], seed=71)
    bt = lay.block_tables.copy()
    bt[0, 1] = lay.num_blocks + 1000
    pkv.get_device_errors(reset=True)
    pkv.paged_decode_attn(dev(val.q), dev(val.k_cache), dev(val.v_cache), dev(bt),
                          dev(lay.context_lens), lay.max_context_len, lay.scale)
    assert pkv.get_device_errors() & pkv.DEVERR_BLOCK_RANGE


def test_decode_context_beyond_table_is_flagged():
    lay, val = _host_case([300, 40], seed=72)
    ctx = lay.context_lens.copy()
    ctx[1] = 5000       # 2 table entries of 256 cannot hold it
    pkv.get_device_errors(reset=True)
    pkv.paged_decode_attn(dev(val.q), dev(val.k_cache), dev(val.v_cache),
                          dev(lay.block_tables), dev(ctx), 5000, lay.scale)
    assert pkv.get_device_errors() & pkv.DEVERR_CONTEXT_RANGE


def test_decode_workspace_too_small_is_rejected():
    lay, val = _host_case([3000, 2000], seed=73)
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attn(dev(val.q), dev(val.k_cache), dev(val.v_cache),
                              dev(lay.block_tables), dev(lay.context_lens), 3000, lay.scale,
                              workspace=ws)
    assert e.value.status == pkv.ERR_WORKSPACE


@pytest.mark.parametrize("n_seqs", [16, 64])
def test_decode_last_tile_every_remainder(n_seqs):
    """A context's last tile is loaded only as far as it holds keys (8-row chunks), so the
    rest of that shared-memory stage keeps whatever an earlier tile left there -- often NaN
    canaries from pool slots past other contexts. Contexts with every remainder 1..64 modulo
    the 64-token tile, on a static grid whose splits merge in clusters (16 sequences) and on
    the work queue (64 sequences: 512 units), must match the oracle."""
    g = w.rng(75)
    ctx = [64 * int(g.integers(0, 11)) + 1 + (i % 64) for i in range(n_seqs)]
    lay, val = _host_case(ctx, seed=76)
    ref = _oracle_step(lay, val)
    out = _gpu_step(lay, dev(val.k_cache), dev(val.v_cache), dev(val.q), dev(val.k_new),
                    dev(val.v_new), 0)
    assert_attention_close(out, ref, f"every last-tile remainder, {n_seqs} sequences")
    assert pkv.get_device_errors() == 0


def test_decode_workspace_counter_left_zero_and_dirty_counter_flagged():
    """With more units than two per SM the CTAs take units from the work counter at the
    start of the workspace, and the CTA that draws last sets it back to zero: calls in a row
    on one workspace need nothing in between. A counter that was not zeroed gives undefined
    results but no fault (a draw below zero ends a CTA's walk); values that a zeroed counter
    cannot give (far past the units, or below zero) set DEVERR_WORKSPACE, and once the
    counter is zeroed again the call is correct."""
    ctx = [700 + 13 * i for i in range(48)]  # 48 sequences x 8 KV heads: 384 units
    lay, val = _host_case(ctx, seed=74)
    oracle.kv_store(val.k_new, val.v_new, lay.slot_mapping, val.k_cache, val.v_cache)
    q, kc, vc = dev(val.q), dev(val.k_cache), dev(val.v_cache)
    bt, cl = dev(lay.block_tables), dev(lay.context_lens)
    ref = oracle.paged_decode(val.q, val.k_cache, val.v_cache, lay.block_tables,
                              lay.context_lens, lay.scale)
    ws = pkv.decode_workspace(lay.batch, 16, 8, 128, lay.max_context_len, 0)
    call = lambda: pkv.paged_decode_attn(q, kc, vc, bt, cl, lay.max_context_len, lay.scale,
                                         workspace=ws)
    pkv.get_device_errors(reset=True)
    for i in range(3):
        assert_attention_close(call(), ref, f"call {i} on the same workspace")
        assert int(ws[:16].count_nonzero()) == 0
    assert pkv.get_device_errors() == 0
    for garbage in (1 << 20, -(1 << 30)):
        ws[:16].view(torch.int32)[0] = garbage
        call()
        torch.cuda.synchronize()
        assert pkv.get_device_errors(reset=True) & pkv.DEVERR_WORKSPACE, garbage
        ws.zero_()
        assert_attention_close(call(), ref, f"zeroed again after a counter of {garbage}")
        assert int(ws[:16].count_nonzero()) == 0
        assert pkv.get_device_errors() == 0


# ------------------------------------------------------------------ full-size workloads
def _full_size(lay, seed, check_rows=None):
    """Device pools drawn on the GPU; the new token stored, decode run with the automatic
    split choice (the benchmark's launch); the oracle on a compact host copy."""
    kc_d, vc_d = fill_sequences_on_device(lay, seed)
    B = lay.batch
    q_d = w.device_bf16_normal((B, 16, 128), seed + 2)
    kn_d = w.device_bf16_normal((B, 8, 128), seed + 3)
    vn_d = w.device_bf16_normal((B, 8, 128), seed + 4)
    out = _gpu_step(lay, kc_d, vc_d, q_d, kn_d, vn_d)
    torch.cuda.synchronize()
    rows = np.arange(B) if check_rows is None else np.asarray(check_rows)
    k_h, v_h, bt = compact_for_oracle(kc_d, vc_d, lay.block_tables[rows])
    ref = oracle.paged_decode(host_bits(q_d)[rows], k_h, v_h, bt, lay.context_lens[rows],
                              lay.scale)
    assert_attention_close(out[torch.from_numpy(rows).cuda()], ref, "full size")
    assert pkv.get_device_errors() == 0


def test_decode_qwen3_batch_full_size():
    """Qwen3-0.6B-shaped decode batch: 256 sequences, contexts U[100, 2048], blocks drawn
    at random from the pool; every output checked."""
    ctx = w.qwen3_decode_lengths()
    lay = w.qwen3_decode_layout(num_blocks=w.blocks_needed(ctx) + 512)
    _full_size(lay, 1000)


def test_decode_long_context_full_size():
    """32 sequences x 32768 tokens; every output checked."""
    lay = w.long_decode_layout(num_blocks=32 * 128 + 64)
    _full_size(lay, 2000)


@pytest.mark.parametrize("batch", [1, 2, 4, 8, 16, 32, 64, 128, 256, 512])
def test_decode_batch_sweep(batch):
    """Batch sweep at context 1024; up to 64 sequences checked per batch."""
    lay = w.sweep_decode_layout(batch, num_blocks=batch * 4 + 16)
    rows = np.arange(batch) if batch <= 64 else w.rng(batch).choice(batch, 64, replace=False)
    _full_size(lay, 3000 + batch, check_rows=np.sort(rows))


def test_decode_on_a_given_stream_without_a_workspace():
    """A call given a stream and no workspace zeroes the workspace it allocates on that
    stream, where the kernel reads its work counter (a queued grid: 48 sequences x 8 KV heads),
    also when the stream is passed as a raw handle."""
    lay, val = _host_case([500 + 7 * i for i in range(48)], seed=77)
    oracle.kv_store(val.k_new, val.v_new, lay.slot_mapping, val.k_cache, val.v_cache)
    ref = oracle.paged_decode(val.q, val.k_cache, val.v_cache, lay.block_tables,
                              lay.context_lens, lay.scale)
    q, kc, vc = dev(val.q), dev(val.k_cache), dev(val.v_cache)
    bt, cl = dev(lay.block_tables), dev(lay.context_lens)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    for handle in (s, s.cuda_stream):
        out = torch.empty_like(q)
        torch.cuda.synchronize()
        pkv.paged_decode_attn(q, kc, vc, bt, cl, lay.max_context_len, lay.scale, out=out,
                              stream=handle)
        s.synchronize()
        assert_attention_close(out, ref, f"stream given as {type(handle).__name__}")
    assert pkv.get_device_errors() == 0


def test_decode_runs_on_the_callers_current_stream():
    """With no stream given, the binding launches on torch's current stream: a side stream's
    handle is what it passes, and a call made under that stream sees the inputs written on it."""
    lay, val = _host_case([300, 1200], seed=59)
    ref = _oracle_step(lay, val)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert pkv._stream(None) == s.cuda_stream
        kc, vc = dev(val.k_cache), dev(val.v_cache)
        out = _gpu_step(lay, kc, vc, dev(val.q), dev(val.k_new), dev(val.v_new))
    s.synchronize()
    assert_attention_close(out, ref, "side stream")
