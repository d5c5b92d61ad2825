"""The decode entry point for callers that cannot allocate device memory.

pkv_paged_decode_attn_noalloc serves callers with no way to get a workspace when they call
decode -- a plug-in in an engine that has given nearly all of HBM to its KV pool and offers
no allocator, or a call site where cudaMalloc is not allowed. Its split results live in a
fixed array inside the library. These tests call it through the C ABI (ctypes on libpkv.so,
and once through the Python wrapper) and check it against the oracle and against the
workspace entry point on the same inputs, within the attention tolerance, on calls in a row:
each call finds the array as the previous one left it. The calls cover the three ways the
array is used: the queued split kernel of the full Qwen3 batch, the one-unit-per-CTA launch
of a small batch (no work counter), and one split (no partial results at all). This file is
named so that pytest collects it after every other test file.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as w
from gpu_util import (assert_attention_close, compact_for_oracle, dev, fill_sequences_on_device,
                      host_bits, host_f64)
from libbuild import build_and_import

pytestmark = pytest.mark.gpu
pkv = build_and_import()
LIB = pkv.lib()
SCRATCH_BYTES = 32 << 20   # PKV_DECODE_NOALLOC_SCRATCH_BYTES in include/pkv.h


def _noalloc(q, kc, vc, bt, ctx, maxc, scale, num_splits, out):
    nb, bs, hkv, d = kc.shape
    B, hq, _ = q.shape
    return LIB.pkv_paged_decode_attn_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kc.data_ptr()),
        ctypes.c_void_p(vc.data_ptr()), ctypes.c_void_p(bt.data_ptr()), bt.shape[1],
        ctypes.c_void_p(ctx.data_ptr()), B, maxc, hq, hkv, d, bs, nb, scale, num_splits,
        ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _tiny_step_on_device():
    """The tiny decode step (contexts {1, 17, 255, 300}): new tokens stored on the device,
    and the oracle's result for the same step."""
    lay, val = w.tiny_decode()
    kc, vc = dev(val.k_cache), dev(val.v_cache)
    pkv.kv_store(dev(val.k_new), dev(val.v_new), dev(lay.slot_mapping), kc, vc)
    kh, vh = val.k_cache.copy(), val.v_cache.copy()
    oracle.kv_store(val.k_new, val.v_new, lay.slot_mapping, kh, vh)
    ref = oracle.paged_decode(val.q, kh, vh, lay.block_tables, lay.context_lens, lay.scale)
    return lay, val, kc, vc, ref


def test_noalloc_matches_oracle_and_workspace_entry_point_on_calls_in_a_row():
    pkv.get_device_errors(reset=True)
    # two calls on the full Qwen3 batch (more units than CTAs: the queued split kernel)
    ctx = w.qwen3_decode_lengths()
    lay = w.qwen3_decode_layout(num_blocks=w.blocks_needed(ctx) + 64)
    assert 0 < pkv.decode_workspace_bytes(lay.batch, 16, 8, 128, lay.max_context_len) <= SCRATCH_BYTES
    kc, vc = fill_sequences_on_device(lay, 7000)
    bt, cl = dev(lay.block_tables), dev(lay.context_lens)
    k_h, v_h, bt_h = compact_for_oracle(kc, vc, lay.block_tables)
    for call, seed in enumerate((7100, 7200)):
        q = w.device_bf16_normal((lay.batch, 16, 128), seed)
        want = pkv.paged_decode_attn(q, kc, vc, bt, cl, lay.max_context_len, lay.scale)
        got = torch.empty_like(q)
        assert _noalloc(q, kc, vc, bt, cl, lay.max_context_len, lay.scale, 0, got) == pkv.OK
        torch.cuda.synchronize()
        assert_attention_close(got, host_f64(want), f"call {call}: workspace entry point")
        ref = oracle.paged_decode(host_bits(q), k_h, v_h, bt_h, lay.context_lens, lay.scale)
        assert_attention_close(got, ref, f"call {call}: oracle")

    # then the tiny step, with the array holding the Qwen3 batch's partials: automatic splits
    # (one unit per CTA, no work counter) through the C ABI, and one split (no partials)
    # through the Python wrapper
    tl, tv, tkc, tvc, tref = _tiny_step_on_device()
    tbt, tcl = dev(tl.block_tables), dev(tl.context_lens)
    tq = dev(tv.q)
    for splits in (0, 1):
        want = pkv.paged_decode_attn(tq, tkc, tvc, tbt, tcl, tl.max_context_len, tl.scale,
                                     num_splits=splits)
        if splits == 0:
            got = torch.full_like(tq, 5.0)
            assert _noalloc(tq, tkc, tvc, tbt, tcl, tl.max_context_len, tl.scale, 0,
                            got) == pkv.OK
        else:
            got = pkv.paged_decode_attn_noalloc(tq, tkc, tvc, tbt, tcl, tl.max_context_len,
                                                tl.scale, num_splits=1)
        torch.cuda.synchronize()
        assert_attention_close(got, tref, f"tiny step, splits={splits}: oracle")
        assert_attention_close(got, host_f64(want), f"tiny step, splits={splits}: workspace")
        # a one-token context returns that token's V exactly
        assert np.array_equal(host_bits(got)[0], np.repeat(tv.logical_v[0][0], 2, axis=0))
    assert pkv.get_device_errors() == 0


def test_noalloc_rejects_plans_larger_than_its_array():
    """32 sequences x 32768 tokens cut into 256 splits need more than the array holds: the
    call is refused before anything runs (the tables only name block 0, and every context is
    1 token, so nothing could be read out of bounds even if it ran)."""
    B, maxc, splits = 32, 32768, 256
    assert pkv.decode_workspace_bytes(B, 16, 8, 128, maxc, splits) > SCRATCH_BYTES
    q = torch.zeros((B, 16, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((4, 256, 8, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((B, 128), dtype=torch.int32, device="cuda")
    cl = torch.ones(B, dtype=torch.int32, device="cuda")
    out = torch.full_like(q, 3.0)
    assert _noalloc(q, kc, kc, bt, cl, maxc, 0.088, splits, out) == pkv.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 3.0).all())
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attn_noalloc(q, kc, kc, bt, cl, maxc, 0.088, num_splits=splits,
                                      out=out)
    assert e.value.status == pkv.ERR_WORKSPACE
