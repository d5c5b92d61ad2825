"""The block manager driving the attention path, as an engine uses it: block tables and slot
mappings come from the library's host block manager, K/V are written with kv_store, and the
attention reads them through the tables.

Six prompts share a 512-token prefix (two 256-token blocks). The first is prefilled in full;
the other five find the two prefix blocks in the cache (512 cached tokens each), so only their
suffix K/V are stored and their prefill queries are the suffix tokens. Then every sequence
decodes one token (may_append takes a new block where the token starts one). Each attention
result is compared with the oracle on the sequences' packed K/V; at the end every block is
free again.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as w
from gpu_util import assert_attention_close, dev, host_bits
from libbuild import build_and_import

pytestmark = pytest.mark.gpu
pkv = build_and_import()

HQ, HKV, D, BS = 16, 8, 128, 256
SCALE = 128 ** -0.5


def _slots(table, positions):
    return np.array([table[p // BS] * BS + p % BS for p in positions], np.int64)


def test_block_manager_prefix_prefill_then_decode():
    g = w.rng(41)
    prefix = g.integers(0, 50000, 512).tolist()
    suffix_lens = [100, 300, 1, 256, 511, 700]
    tokens = [prefix + g.integers(0, 50000, s).tolist() for s in suffix_lens]
    nb = 40
    bm = pkv.BlockManager(nb, BS)
    kc = torch.zeros((nb, BS, HKV, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    # K/V of every token of every sequence; the prefix's are shared (same tokens, same K/V)
    pk, pv = w.host_bf16_normal(g, (512, HKV, D)), w.host_bf16_normal(g, (512, HKV, D))
    keys, vals = [], []
    for s in suffix_lens:
        keys.append(np.concatenate([pk, w.host_bf16_normal(g, (s, HKV, D))]))
        vals.append(np.concatenate([pv, w.host_bf16_normal(g, (s, HKV, D))]))

    tables, cached = [], []
    for i, toks in enumerate(tokens):
        t, c = bm.allocate(toks)
        tables.append(t)
        cached.append(c)
        assert c == (0 if i == 0 else 512)
        assert t[:2] == tables[0][:2]                      # the shared prefix blocks
        new = range(c, len(toks))                          # tokens whose K/V are not cached
        pkv.kv_store(dev(keys[i][c:]), dev(vals[i][c:]), dev(_slots(t, new)), kc, vc)
    assert bm.ref_count(tables[0][0]) == 6 and bm.ref_count(tables[0][1]) == 6

    # prefill: sequence 0 in full, the others only their suffixes, keys through the tables
    lens_k = np.array([len(t) for t in tokens], np.int32)
    lens_q = lens_k - np.array(cached, np.int32)
    cq = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    W = max(len(t) for t in tables) + 1
    bt = np.full((len(tokens), W), -1, np.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
    q = w.host_bf16_normal(g, (int(lens_q.sum()), HQ, D))
    out = pkv.varlen_prefill_attn(dev(q), kc, vc, dev(cq), dev(ck), int(lens_q.max()),
                                  int(lens_k.max()), SCALE, block_table=dev(bt))
    ref = oracle.varlen_prefill(q, np.concatenate(keys), np.concatenate(vals), cq, ck, SCALE)
    assert_attention_close(out, ref, "prefill through the block manager's tables")

    # one decode step: append a token to every sequence
    knew, vnew = [], []
    for i in range(len(tokens)):
        tokens[i].append(int(g.integers(0, 50000)))
        assert bm.can_append(len(tokens[i]))
        tables[i] = bm.may_append(tokens[i], tables[i])
        knew.append(w.host_bf16_normal(g, (1, HKV, D)))
        vnew.append(w.host_bf16_normal(g, (1, HKV, D)))
        keys[i] = np.concatenate([keys[i], knew[-1]])
        vals[i] = np.concatenate([vals[i], vnew[-1]])
    assert len(tables[3]) == 4                           # 768 -> 769 tokens: a new block
    assert [len(t) for t in tables] == [3, 4, 3, 4, 4, 5]
    slots = np.concatenate([_slots(tables[i], [len(tokens[i]) - 1]) for i in range(len(tokens))])
    pkv.kv_store(dev(np.concatenate(knew)), dev(np.concatenate(vnew)), dev(slots), kc, vc)
    ctx = np.array([len(t) for t in tokens], np.int32)
    bt = np.full((len(tokens), W + 1), -1, np.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
    qd = w.host_bf16_normal(g, (len(tokens), HQ, D))
    out = pkv.paged_decode_attn(dev(qd), kc, vc, dev(bt), dev(ctx), int(ctx.max()), SCALE)
    ref = oracle.paged_decode(qd, host_bits(kc), host_bits(vc), bt, ctx, SCALE)
    assert_attention_close(out, ref, "decode through the block manager's tables")
    # the same decode from the packed K/V (the pool holds exactly the sequences' K/V)
    for i in range(len(tokens)):
        r = oracle.varlen_prefill(qd[i:i + 1], keys[i], vals[i], np.array([0, 1], np.int32),
                                  np.array([0, ctx[i]], np.int32), SCALE)
        assert_attention_close(out[i:i + 1], r, f"decode row {i} vs packed")

    for t in tables:
        bm.deallocate(t)
    assert bm.num_free == nb
    assert pkv.get_device_errors() == 0
