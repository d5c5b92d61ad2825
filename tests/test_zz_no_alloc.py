"""The decode entry point for callers that cannot allocate device memory.

pkv_paged_decode_attn_noalloc serves callers with no way to get a workspace when they call
decode -- a plug-in in an engine that has given nearly all of HBM to its KV pool and offers
no allocator, or a call site where cudaMalloc is not allowed. Its split results live in a
fixed array inside the library. These tests call it through the C ABI (ctypes on libpkv.so)
and check it against the workspace entry point on the same inputs, within the attention
tolerance, on two calls in a row (the second call reuses the array the first one left
behind). This file is named so that pytest collects it after every other test file.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as w
from gpu_util import assert_attention_close, dev, fill_sequences_on_device, host_f64
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


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    pkv.get_device_errors(reset=True)
    ctx = w.qwen3_decode_lengths()
    lay = w.qwen3_decode_layout(num_blocks=w.blocks_needed(ctx) + 64)
    assert 0 < pkv.decode_workspace_bytes(lay.batch, 16, 8, 128, lay.max_context_len) <= SCRATCH_BYTES
    kc, vc = fill_sequences_on_device(lay, 7000)
    bt, cl = dev(lay.block_tables), dev(lay.context_lens)
    for call, seed in enumerate((7100, 7200)):
        q = w.device_bf16_normal((lay.batch, 16, 128), seed)
        want = pkv.paged_decode_attn(q, kc, vc, bt, cl, lay.max_context_len, lay.scale)
        got = torch.empty_like(q)
        assert _noalloc(q, kc, vc, bt, cl, lay.max_context_len, lay.scale, 0, got) == pkv.OK
        torch.cuda.synchronize()
        assert_attention_close(got, host_f64(want), f"call {call}")
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
