"""pkv_paged_decode_step (the new tokens stored inside the decode kernel) against the two-call
path (pkv_kv_store, then pkv_paged_decode_attn): the same output and the same pool, bit for
bit, for every GQA grouping (groups of 1 and 2 take the fused path, 3 and 4 the store kernel
first), split settings, padding rows (slot -1, context 0), new K/V given as strided views of a
fused projection, and the full Qwen3 decode batch; plus the oracle on the tiny step and on
the full Qwen3 batch.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as w
from gpu_util import (assert_attention_close, compact_for_oracle, dev, fill_sequences_on_device,
                      host_bits, remap_slots)
from libbuild import build_and_import

pytestmark = pytest.mark.gpu
pkv = build_and_import()


def _both(lay, kc, vc, q, kn, vn, num_splits=0):
    """Output and pools of the fused step and of store-then-decode, on copies of the pools."""
    slots, tables, ctx = dev(lay.slot_mapping), dev(lay.block_tables), dev(lay.context_lens)
    kc2, vc2 = kc.clone(), vc.clone()
    fused = pkv.paged_decode_step(q, kn, vn, slots, kc, vc, tables, ctx, lay.max_context_len,
                                  lay.scale, num_splits=num_splits)
    pkv.kv_store(kn, vn, slots, kc2, vc2)
    two = pkv.paged_decode_attn(q, kc2, vc2, tables, ctx, lay.max_context_len, lay.scale,
                                num_splits=num_splits)
    return fused, two, (kc, vc), (kc2, vc2)


def _same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def _case(ctx, seed, hq=16, hkv=8):
    g = w.rng(seed)
    lay = w.decode_layout(np.asarray(ctx, np.int32), w.blocks_needed(ctx) + 3, g,
                          num_q_heads=hq, num_kv_heads=hkv)
    val = w.decode_values(lay, g)
    return lay, val


def test_tiny_step_matches_two_calls_and_oracle():
    lay, val = w.tiny_decode()
    kc, vc = dev(val.k_cache), dev(val.v_cache)
    fused, two, pf, pt = _both(lay, kc, vc, dev(val.q), dev(val.k_new), dev(val.v_new))
    assert _same(fused, two) and _same(pf[0], pt[0]) and _same(pf[1], pt[1])
    kh, vh = val.k_cache.copy(), val.v_cache.copy()
    oracle.kv_store(val.k_new, val.v_new, lay.slot_mapping, kh, vh)
    ref = oracle.paged_decode(val.q, kh, vh, lay.block_tables, lay.context_lens, lay.scale)
    assert_attention_close(fused, ref, "tiny step")
    assert pkv.get_device_errors() == 0


@pytest.mark.parametrize("hq,hkv", [(16, 8), (8, 8), (12, 4), (16, 4)])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_groupings_and_splits(hq, hkv, num_splits):
    ctx = [1, 2, 63, 64, 65, 255, 256, 257, 700, 1500]
    lay, val = _case(ctx, seed=hq * 10 + hkv + num_splits, hq=hq, hkv=hkv)
    fused, two, pf, pt = _both(lay, dev(val.k_cache), dev(val.v_cache), dev(val.q),
                               dev(val.k_new), dev(val.v_new), num_splits)
    assert _same(fused, two), "output"
    assert _same(pf[0], pt[0]) and _same(pf[1], pt[1]), "pools"
    assert pkv.get_device_errors() == 0


def test_padding_rows_and_strided_new_kv():
    """Rows 3 and 7 are padding (context 0, slot -1); k_new and v_new are column slices of a
    fused [B, (Hq + 2 Hkv) * D] buffer."""
    ctx = [5, 300, 1, 0, 129, 2000, 64, 0]
    g = w.rng(61)
    lay = w.decode_layout(np.asarray(ctx, np.int32), w.blocks_needed(ctx) + 3, g)
    lay.slot_mapping[np.asarray(ctx) == 0] = -1
    val = w.decode_values(lay, g)
    B, hq, hkv, d = len(ctx), 16, 8, 128
    qkv = torch.zeros((B, (hq + 2 * hkv) * d), dtype=torch.bfloat16, device="cuda")
    qkv[:, hq * d:(hq + hkv) * d] = dev(val.k_new).reshape(B, -1)
    qkv[:, (hq + hkv) * d:] = dev(val.v_new).reshape(B, -1)
    kn = qkv[:, hq * d:(hq + hkv) * d].view(B, hkv, d)
    vn = qkv[:, (hq + hkv) * d:].view(B, hkv, d)
    fused, two, pf, pt = _both(lay, dev(val.k_cache), dev(val.v_cache), dev(val.q), kn, vn)
    assert _same(fused, two) and _same(pf[0], pt[0]) and _same(pf[1], pt[1])
    assert not fused[np.asarray(ctx) == 0].view(torch.int16).any()
    assert pkv.get_device_errors() == 0


def test_full_qwen3_batch():
    """The benchmark's decode batch (256 sequences, contexts U[100, 2048]) with the automatic
    split choice: fused step == store + decode, bit for bit; and the fused step against the
    oracle, which stores the same new tokens into its own copy of the referenced blocks and
    attends over them (every output compared, the stored blocks bit for bit)."""
    lens = w.qwen3_decode_lengths()
    lay = w.qwen3_decode_layout(num_blocks=w.blocks_needed(lens) + 64)
    kc, vc = fill_sequences_on_device(lay, 71)
    q = w.device_bf16_normal((lay.batch, 16, 128), 72)
    kn = w.device_bf16_normal((lay.batch, 8, 128), 73)
    vn = w.device_bf16_normal((lay.batch, 8, 128), 74)
    k_h, v_h, bt_h = compact_for_oracle(kc, vc, lay.block_tables)   # before the step
    fused, two, pf, pt = _both(lay, kc, vc, q, kn, vn)
    assert _same(fused, two)
    assert _same(pf[0], pt[0]) and _same(pf[1], pt[1])
    assert pkv.get_device_errors() == 0
    oracle.kv_store(host_bits(kn), host_bits(vn),
                    remap_slots(lay.block_tables, lay.slot_mapping, lay.block_size), k_h, v_h)
    ref = oracle.paged_decode(host_bits(q), k_h, v_h, bt_h, lay.context_lens, lay.scale)
    assert_attention_close(fused, ref, "full Qwen3 batch: oracle")
    k_after, v_after, _ = compact_for_oracle(pf[0], pf[1], lay.block_tables)
    assert np.array_equal(k_after, k_h) and np.array_equal(v_after, v_h), "stored rows"
