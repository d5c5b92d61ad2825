"""Varlen causal prefill on the GPU (tcgen05 path) against the oracle, through the C ABI.

Element-wise parity within |err| <= 1e-2 + 1e-2 |ref| at small ragged sizes (tiles of 128
rows and keys with partial tails, several sequences, every supported GQA grouping), in both
key layouts (packed, and the paged pool through block_table); the full varlen workload and
the prefix-cached workload on sampled sequences; and the invariants: paged == packed and
shared prefix blocks == private copies, bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as w
from gpu_util import assert_attention_close, canary_pool, dev, host_bits
from libbuild import build_and_import

pytestmark = pytest.mark.gpu
pkv = build_and_import()


def _case(lens_q, seed, hq=16, hkv=8, lens_k=None, nb_spare=4):
    g = w.rng(seed)
    lens_q = np.asarray(lens_q, np.int32)
    lens_k = lens_q if lens_k is None else np.asarray(lens_k, np.int32)
    Tq, Tk = int(lens_q.sum()), int(lens_k.sum())
    q = w.host_bf16_normal(g, (Tq, hq, 128))
    k = w.host_bf16_normal(g, (Tk, hkv, 128))
    v = w.host_bf16_normal(g, (Tk, hkv, 128))
    cq = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    return q, k, v, cq, ck


def _run(q, k, v, cq, ck, causal=True, block_table=None, scale=128 ** -0.5, q_dev=None):
    lq = np.diff(cq)
    lk = np.diff(ck)
    return pkv.varlen_prefill_attn(dev(q) if q_dev is None else q_dev, dev(k), dev(v), dev(cq),
                                   dev(ck), int(lq.max()), int(lk.max()), scale, causal=causal,
                                   block_table=None if block_table is None else dev(block_table))


@pytest.mark.parametrize("lens", [[1], [5, 64, 65], [127, 128, 129], [300, 1, 200, 511],
                                  [1024, 3, 700]])
def test_prefill_packed_causal(lens):
    q, k, v, cq, ck = _case(lens, seed=sum(lens))
    ref = oracle.varlen_prefill(q, k, v, cq, ck, 128 ** -0.5)
    assert_attention_close(_run(q, k, v, cq, ck), ref, f"lens={lens}")
    assert pkv.get_device_errors() == 0


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 4), (16, 2), (32, 8)])
def test_prefill_head_groupings(hq, hkv):
    q, k, v, cq, ck = _case([130, 67, 256], seed=hq * 10 + hkv, hq=hq, hkv=hkv)
    ref = oracle.varlen_prefill(q, k, v, cq, ck, 128 ** -0.5)
    assert_attention_close(_run(q, k, v, cq, ck), ref, f"hq={hq} hkv={hkv}")


def test_prefill_out_aligned_to_16_bytes_only():
    """An out buffer that starts 16 bytes past a 32-byte boundary takes the 16-byte store
    path: the same values as an aligned out, bit for bit, and no byte outside it written."""
    q, k, v, cq, ck = _case([300, 5, 129], seed=41)
    aligned = _run(q, k, v, cq, ck)
    n = aligned.numel()
    big = torch.full((n + 32,), -7.0, dtype=torch.bfloat16, device="cuda")
    out = big[8:8 + n].view(aligned.shape)  # 8 bf16 = 16 bytes past the start
    assert out.data_ptr() % 32 == 16
    lq = np.diff(cq)
    pkv.varlen_prefill_attn(dev(q), dev(k), dev(v), dev(cq), dev(ck), int(lq.max()),
                            int(lq.max()), 128 ** -0.5, out=out)
    assert torch.equal(out.view(torch.int16), aligned.view(torch.int16))
    assert (big[:8] == -7.0).all() and (big[8 + n:] == -7.0).all()
    assert pkv.get_device_errors() == 0


def test_prefill_non_causal_and_unequal_lengths():
    q, k, v, cq, ck = _case([100, 37], seed=5, lens_k=[300, 129])
    for causal in (False, True):
        ref = oracle.varlen_prefill(q, k, v, cq, ck, 0.1, causal=causal)
        assert_attention_close(_run(q, k, v, cq, ck, causal=causal, scale=0.1), ref,
                               f"causal={causal}")


def test_prefill_more_queries_than_keys_gives_zero_rows():
    q, k, v, cq, ck = _case([200, 10], seed=6, lens_k=[70, 10])
    ref = oracle.varlen_prefill(q, k, v, cq, ck, 128 ** -0.5)
    out = _run(q, k, v, cq, ck)
    assert_attention_close(out, ref, "Lq > Lk")
    assert not host_bits(out)[:130].any()      # queries 0..129 of sequence 0 see no key


def test_prefill_empty_sequences_in_batch():
    q, k, v, cq, ck = _case([0, 50, 0, 129], seed=7)
    ref = oracle.varlen_prefill(q, k, v, cq, ck, 128 ** -0.5)
    assert_attention_close(_run(q, k, v, cq, ck), ref, "empty sequences")


def test_prefill_q_as_view_of_fused_qkv():
    g = w.rng(8)
    lens = np.array([90, 260], np.int32)
    T = int(lens.sum())
    qkv = w.host_bf16_normal(g, (T, (16 + 16) * 128))
    q = qkv[:, :16 * 128].reshape(T, 16, 128)
    k = qkv[:, 16 * 128:24 * 128].reshape(T, 8, 128)
    v = qkv[:, 24 * 128:].reshape(T, 8, 128)
    cq = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    qkv_d = dev(qkv)
    out = pkv.varlen_prefill_attn(qkv_d[:, :16 * 128].view(T, 16, 128),
                                  qkv_d[:, 16 * 128:24 * 128].view(T, 8, 128),
                                  qkv_d[:, 24 * 128:].view(T, 8, 128), dev(cq), dev(cq), 260, 260,
                                  128 ** -0.5)
    ref = oracle.varlen_prefill(q, k, v, cq, cq, 128 ** -0.5)
    assert_attention_close(out, ref, "fused qkv views")


def _paged(lens, seed, canary_tail=True):
    """Prompts stored into a paged pool via slot_mapping (pool slots past each prompt keep a
    NaN canary), read back through block_table."""
    g = w.rng(seed)
    lay = w.prefill_layout(lens, w.blocks_needed(lens) + 5, g)
    val = w.prefill_values(lay, g)
    kc, vc = val.k_cache.copy(), val.v_cache.copy()
    oracle.kv_store(val.k, val.v, lay.slot_mapping, kc, vc)
    return lay, val, kc, vc


def test_prefill_paged_matches_oracle_and_packed_bitwise():
    lay, val, kc, vc = _paged([300, 129, 513, 1], seed=9)
    cq = lay.cu_seqlens_q
    ref = oracle.varlen_prefill(val.q, kc, vc, cq, cq, lay.scale, block_table=lay.block_table)
    paged = _run(val.q, kc, vc, cq, cq, block_table=lay.block_table)
    packed = _run(val.q, val.k, val.v, cq, cq)
    assert_attention_close(paged, ref, "paged")
    assert np.array_equal(host_bits(paged), host_bits(packed))


def test_prefill_paged_store_then_attend_on_device():
    """The prefill step as the engine runs it: kv_store of the prompt's K/V into the pool,
    then attention through block_table, all on the device."""
    lay, val, _, _ = _paged([700, 45], seed=10)
    kc_d, vc_d = dev(val.k_cache), dev(val.v_cache)
    pkv.kv_store(dev(val.k), dev(val.v), dev(lay.slot_mapping), kc_d, vc_d)
    cq = lay.cu_seqlens_q
    out = pkv.varlen_prefill_attn(dev(val.q), kc_d, vc_d, dev(cq), dev(cq), 700, 700, lay.scale,
                                  block_table=dev(lay.block_table))
    ref = oracle.varlen_prefill(val.q, val.k, val.v, cq, cq, lay.scale)
    assert_attention_close(out, ref, "store + paged prefill")


def _prefix(suffix, seed, private=False, prefix_len=512):
    g = w.rng(seed)
    nb = 3 * len(suffix) + 8 + (len(suffix) * prefix_len // 256 if private else prefix_len // 256)
    lay = w.prefix_prefill_layout(suffix, prefix_len, nb, g, private_prefix=private)
    val = w.prefill_values(lay, w.rng(seed + 1))
    kc, vc = val.k_cache.copy(), val.v_cache.copy()
    rows = w.suffix_rows(lay)
    oracle.kv_store(val.k[rows], val.v[rows], lay.slot_mapping, kc, vc)
    return lay, val, kc, vc


def test_prefix_cached_prefill_small():
    lay, val, kc, vc = _prefix([256, 300, 1, 129], seed=11)
    ref = oracle.varlen_prefill(val.q, kc, vc, lay.cu_seqlens_q, lay.cu_seqlens_k, lay.scale,
                                block_table=lay.block_table)
    out = _run(val.q, kc, vc, lay.cu_seqlens_q, lay.cu_seqlens_k, block_table=lay.block_table)
    assert_attention_close(out, ref, "prefix cached")
    # the cached computation gives the suffix rows of the uncached one
    ck = lay.cu_seqlens_k
    rows = w.suffix_rows(lay)
    q_full = np.zeros((int(ck[-1]), 16, 128), np.uint16)
    q_full[rows] = val.q
    full = _run(q_full, val.k, val.v, ck, ck)
    assert_attention_close(full[torch.from_numpy(rows).cuda()], ref, "uncached rows")


def test_prefix_shared_blocks_equal_private_copies_bitwise():
    a = _prefix([200, 333, 64], seed=12)
    b = _prefix([200, 333, 64], seed=12, private=True)
    outs = [host_bits(_run(val.q, kc, vc, lay.cu_seqlens_q, lay.cu_seqlens_k,
                           block_table=lay.block_table)) for lay, val, kc, vc in (a, b)]
    assert a[0].ref_count.max() == 3 and b[0].ref_count.max() == 1
    assert np.array_equal(outs[0], outs[1])


def test_prefill_bad_block_id_is_flagged():
    lay, val, kc, vc = _paged([300], seed=13)
    bt = lay.block_table.copy()
    bt[0, 1] = -7
    pkv.get_device_errors(reset=True)
    cq = lay.cu_seqlens_q
    _run(val.q, kc, vc, cq, cq, block_table=bt)
    assert pkv.get_device_errors() & pkv.DEVERR_BLOCK_RANGE


def test_prefill_skewed_lengths():
    """One long prompt among many one- to three-token ones: the work list holds only blocks
    that have queries (the long prompt's 20 blocks first), and every row matches the oracle."""
    lens = [2500] + [1, 2, 3] * 40
    q, k, v, cq, ck = _case(lens, seed=29)
    ref = oracle.varlen_prefill(q, k, v, cq, ck, 128 ** -0.5)
    pkv.get_device_errors(reset=True)
    assert_attention_close(_run(q, k, v, cq, ck), ref, "skewed")
    assert pkv.get_device_errors() == 0


def test_prefill_longer_than_max_seqlen_is_flagged():
    """A sequence longer than max_seqlen_q sets the sequence-length error bit (its query
    blocks past the bound are not computed); the other sequences are unaffected."""
    lens = [100, 300]
    q, k, v, cq, ck = _case(lens, seed=31)
    ref = oracle.varlen_prefill(q, k, v, cq, ck, 128 ** -0.5)
    pkv.get_device_errors(reset=True)
    out = pkv.varlen_prefill_attn(dev(q), dev(k), dev(v), dev(cq), dev(ck), 128, 300,
                                  128 ** -0.5)
    assert pkv.get_device_errors() & pkv.DEVERR_SEQLEN_RANGE
    assert_attention_close(out[:100], ref[:100], "the sequence within the bound")
    pkv.get_device_errors(reset=True)


# ------------------------------------------------------------------ full-size workloads
def _sampled_oracle(q_d, k_d, v_d, cq, ck, seqs, block_table=None, kc_d=None, vc_d=None):
    """Oracle on a few sequences, taking their rows back from the device."""
    outs = []
    for n in seqs:
        a, b = int(cq[n]), int(cq[n + 1])
        qn = host_bits(q_d[a:b])
        if block_table is None:
            c, d = int(ck[n]), int(ck[n + 1])
            kn, vn = host_bits(k_d[c:d]), host_bits(v_d[c:d])
            cqn = np.array([0, b - a], np.int32)
            ckn = np.array([0, d - c], np.int32)
            outs.append(oracle.varlen_prefill(qn, kn, vn, cqn, ckn, 128 ** -0.5))
        else:
            lk = int(ck[n + 1] - ck[n])
            blocks = block_table[n, :-(-lk // 256)]
            idt = torch.from_numpy(blocks.astype(np.int64)).cuda()
            kn, vn = host_bits(kc_d[idt]), host_bits(vc_d[idt])
            bt = np.arange(len(blocks), dtype=np.int32)[None]
            outs.append(oracle.varlen_prefill(qn, kn, vn, np.array([0, b - a], np.int32),
                                              np.array([0, lk], np.int32), 128 ** -0.5,
                                              block_table=bt))
    return outs


def _per_quartile(lens, per, seed):
    """The longest and the shortest sequence, and `per` random sequences from each quartile
    of the lengths."""
    order = np.argsort(lens, kind="stable")
    g = w.rng(seed)
    picked = {int(order[0]), int(order[-1])}
    for part in np.array_split(order, 4):
        picked.update(int(x) for x in g.choice(part, per, replace=False))
    return sorted(picked)


def test_prefill_varlen_full_size():
    """Varlen causal prefill: 256 prompts U[100, 1024] (~143k tokens), packed; the longest,
    the shortest and four random prompts of each length quartile checked against the
    oracle (18 of 256)."""
    lens = w.varlen_prefill_lengths()
    cq = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cq[-1])
    q_d = w.device_bf16_normal((T, 16, 128), 401)
    k_d = w.device_bf16_normal((T, 8, 128), 402)
    v_d = w.device_bf16_normal((T, 8, 128), 403)
    out = pkv.varlen_prefill_attn(q_d, k_d, v_d, dev(cq), dev(cq), int(lens.max()),
                                  int(lens.max()), 128 ** -0.5)
    seqs = _per_quartile(lens, 4, 77)
    refs = _sampled_oracle(q_d, k_d, v_d, cq, cq, seqs)
    for n, ref in zip(seqs, refs):
        assert_attention_close(out[int(cq[n]):int(cq[n + 1])], ref, f"seq {n}")
    assert pkv.get_device_errors() == 0


def test_prefix_prefill_full_size():
    """Prefix-cached prefill: 64 sequences sharing a 2048-token prefix (8 ref-counted blocks),
    suffixes U[256, 768]; queries are the suffixes, keys come through block_table. The
    longest, the shortest and two random suffixes of each length quartile checked against
    the oracle (10 of 64)."""
    lay = w.prefix_prefill_case_layout(num_blocks=8 + 64 * 3 + 32)
    assert lay.ref_count.max() == 64
    bs = 256
    kc_d = canary_pool(lay.num_blocks, bs, 8, 128)
    vc_d = canary_pool(lay.num_blocks, bs, 8, 128)
    shared = torch.from_numpy(lay.block_table[0, :8].astype(np.int64)).cuda()
    kc_d[shared] = w.device_bf16_normal((8, bs, 8, 128), 501)
    vc_d[shared] = w.device_bf16_normal((8, bs, 8, 128), 502)
    Tq = int(lay.seqlens_q.sum())
    pkv.kv_store(w.device_bf16_normal((Tq, 8, 128), 503), w.device_bf16_normal((Tq, 8, 128), 504),
                 dev(lay.slot_mapping), kc_d, vc_d)
    q_d = w.device_bf16_normal((Tq, 16, 128), 505)
    cq, ck = lay.cu_seqlens_q, lay.cu_seqlens_k
    out = pkv.varlen_prefill_attn(q_d, kc_d, vc_d, dev(cq), dev(ck), int(lay.seqlens_q.max()),
                                  int(lay.seqlens_k.max()), 128 ** -0.5,
                                  block_table=dev(lay.block_table))
    seqs = _per_quartile(lay.seqlens_q, 2, 78)
    refs = _sampled_oracle(q_d, None, None, cq, ck, seqs, block_table=lay.block_table,
                           kc_d=kc_d, vc_d=vc_d)
    for n, ref in zip(seqs, refs):
        assert_attention_close(out[int(cq[n]):int(cq[n + 1])], ref, f"seq {n}")
    assert pkv.get_device_errors() == 0


def test_prefill_one_32k_prompt_sampled_rows():
    """One causal prompt of 32768 tokens (256 query blocks of 128, the longest rows read 256 key
    tiles); sampled query rows checked against the oracle, each as a one-query sequence over
    the keys up to its position (the bottom-right alignment makes that query see exactly
    keys 0 .. p)."""
    L = 32768
    q_d = w.device_bf16_normal((L, 16, 128), 611)
    k_d = w.device_bf16_normal((L, 8, 128), 612)
    v_d = w.device_bf16_normal((L, 8, 128), 613)
    cq = np.array([0, L], np.int32)
    out = pkv.varlen_prefill_attn(q_d, k_d, v_d, dev(cq), dev(cq), L, L, 128 ** -0.5)
    for p in (0, 1, 127, 128, 4095, 16384, 30000, L - 1):
        qn = host_bits(q_d[p:p + 1])
        kn, vn = host_bits(k_d[:p + 1]), host_bits(v_d[:p + 1])
        ref = oracle.varlen_prefill(qn, kn, vn, np.array([0, 1], np.int32),
                                    np.array([0, p + 1], np.int32), 128 ** -0.5)
        assert_attention_close(out[p:p + 1], ref, f"row {p}")
    assert pkv.get_device_errors() == 0


def test_prefill_three_thousand_tiny_prompts():
    """3000 prompts of 1 .. 40 tokens: the planning kernel's count, rank and fill loops take
    several passes over its 1024 threads; every row checked against the oracle."""
    g = w.rng(620)
    lens = g.integers(1, 41, 3000)
    q, k, v, cq, ck = _case(lens, seed=621)
    ref = oracle.varlen_prefill(q, k, v, cq, ck, 128 ** -0.5)
    assert_attention_close(_run(q, k, v, cq, ck), ref, "3000 tiny prompts")
    assert pkv.get_device_errors() == 0
