"""Chunked prefill through the block table: a long prompt is prefilled in pieces, each piece
storing its K/V into the pool (kv_store) and then attending, through block_table, to every key
stored so far (the cached earlier pieces plus itself, with the causal mask aligned to the end
of the keys). This is how the scheduler of «nano-vLLM 最小化vLLM重新实现» (架构 2) prefills
the first sequence in chunks, and how its attention takes a block_table with cached blocks
(架构 5).

Pieces that start at multiples of 128 queries give the same bits as one prefill of the whole
prompt (the kernel's rows are grouped in 128-row tiles and every row walks the same key tiles
in the same order); ragged pieces match the oracle within the attention tolerance. A batch
that mixes one piece of a long prompt with whole short prompts matches the oracle too.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as w
from gpu_util import assert_attention_close, dev
from libbuild import build_and_import

pytestmark = pytest.mark.gpu
pkv = build_and_import()

HQ, HKV, D, BS = 16, 8, 128, 256
SCALE = 128 ** -0.5


def _prompt(L, seed, nb_spare=3):
    g = w.rng(seed)
    nblk = -(-L // BS)
    blocks = g.permutation(nblk + nb_spare)[:nblk].astype(np.int32)
    q = w.host_bf16_normal(g, (L, HQ, D))
    k = w.host_bf16_normal(g, (L, HKV, D))
    v = w.host_bf16_normal(g, (L, HKV, D))
    nb = nblk + nb_spare
    return q, k, v, blocks, nb


def _chunked(q, k, v, blocks, nb, cuts):
    """Prefill the prompt piece by piece; returns the concatenated outputs."""
    kc = torch.zeros((nb, BS, HKV, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    bt = dev(blocks[None, :])
    outs = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        pos = np.arange(a, b)
        slots = (blocks[pos // BS].astype(np.int64) * BS + pos % BS)
        pkv.kv_store(dev(k[a:b]), dev(v[a:b]), dev(slots), kc, vc)
        cq = dev(np.array([0, b - a], np.int32))
        ck = dev(np.array([0, b], np.int32))
        outs.append(pkv.varlen_prefill_attn(dev(q[a:b]), kc, vc, cq, ck, b - a, b, SCALE,
                                            block_table=bt))
    return torch.cat(outs)


@pytest.mark.parametrize("L,chunk", [(2000, 512), (1500, 128), (1100, 384)])
def test_aligned_chunks_equal_one_prefill_bitwise(L, chunk):
    q, k, v, blocks, nb = _prompt(L, seed=L + chunk)
    cuts = list(range(0, L, chunk)) + [L]
    got = _chunked(q, k, v, blocks, nb, cuts)
    whole = _chunked(q, k, v, blocks, nb, [0, L])
    assert torch.equal(got.view(torch.int16), whole.view(torch.int16))
    ref = oracle.varlen_prefill(q, k, v, np.array([0, L], np.int32), np.array([0, L], np.int32),
                                SCALE)
    assert_attention_close(got, ref, f"L={L} chunk={chunk}")
    assert pkv.get_device_errors() == 0


@pytest.mark.parametrize("cuts", [[0, 300, 301, 900, 1234], [0, 1, 2, 3, 700], [0, 255, 256, 257, 600]])
def test_ragged_chunks_match_oracle(cuts):
    L = cuts[-1]
    q, k, v, blocks, nb = _prompt(L, seed=sum(cuts))
    got = _chunked(q, k, v, blocks, nb, cuts)
    ref = oracle.varlen_prefill(q, k, v, np.array([0, L], np.int32), np.array([0, L], np.int32),
                                SCALE)
    assert_attention_close(got, ref, f"cuts={cuts}")
    assert pkv.get_device_errors() == 0


def test_mixed_batch_chunk_with_whole_prompts():
    """One varlen call: the second piece (queries 700..1300) of a 1300-token prompt whose first
    700 tokens are already in the pool, together with three whole short prompts."""
    g = w.rng(77)
    long_q, long_k, long_v, _, _ = _prompt(1300, seed=78)
    shorts = [37, 256, 400]
    lens_k = [1300] + shorts
    lens_q = [600] + shorts
    nblk = [-(-L // BS) for L in lens_k]
    nb = sum(nblk) + 4
    perm = g.permutation(nb).astype(np.int32)
    tables, o = [], 0
    for n in nblk:
        tables.append(perm[o:o + n])
        o += n
    W = max(nblk)
    bt = np.full((4, W), -1, np.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
    qs = [long_q[700:]] + [w.host_bf16_normal(g, (L, HQ, D)) for L in shorts]
    ks = [long_k] + [w.host_bf16_normal(g, (L, HKV, D)) for L in shorts]
    vs = [long_v] + [w.host_bf16_normal(g, (L, HKV, D)) for L in shorts]
    kc = torch.zeros((nb, BS, HKV, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    for i in range(4):
        pos = np.arange(lens_k[i])
        slots = tables[i][pos // BS].astype(np.int64) * BS + pos % BS
        pkv.kv_store(dev(ks[i]), dev(vs[i]), dev(slots), kc, vc)
    cq = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    q = np.concatenate(qs)
    out = pkv.varlen_prefill_attn(dev(q), kc, vc, dev(cq), dev(ck), max(lens_q), max(lens_k),
                                  SCALE, block_table=dev(bt))
    ref = oracle.varlen_prefill(q, np.concatenate(ks), np.concatenate(vs), cq, ck, SCALE)
    assert_attention_close(out, ref, "mixed batch")
    # the piece's rows equal the same rows of a prefill of the whole long prompt
    whole = oracle.varlen_prefill(long_q, long_k, long_v, np.array([0, 1300], np.int32),
                                  np.array([0, 1300], np.int32), SCALE)
    assert_attention_close(out[:600], whole[700:], "piece vs whole prompt")
    assert pkv.get_device_errors() == 0
