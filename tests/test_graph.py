"""A decode step (kv_store of the new tokens, then paged decode attention) captured once in a
CUDA graph per batch bucket and replayed over several steps, as a serving engine runs decode.

The graph is captured with fixed device buffers (queries, new K/V, slot mapping, block table,
context lengths, workspace, output) sized for the bucket and for a maximum context length;
each replay reads whatever the buffers hold. Rows past the live batch are padding: context
length 0 and slot -1, so nothing is stored for them and their output is zero. Every replay is
compared with the oracle element by element, and with an eager call of the same arguments
bit for bit.
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
CAP = 4096            # the longest context any captured step may see
STEPS = 3


def _slots(tables, ctx):
    s = np.full(len(ctx), -1, np.int64)
    for b, c in enumerate(ctx):
        if c > 0:
            s[b] = int(tables[b, (c - 1) // BS]) * BS + (c - 1) % BS
    return s


@pytest.mark.parametrize("bucket,live", [(1, 1), (4, 3), (16, 11), (64, 64)])
def test_decode_step_graph_replay(bucket, live):
    g = w.rng(900 + bucket)
    final = g.integers(3, 2000, size=live).astype(np.int32)
    lay = w.decode_layout(final, w.blocks_needed(final) + 4, g, num_q_heads=HQ,
                          num_kv_heads=HKV, table_width=CAP // BS)
    val = w.decode_values(lay, g)
    W = lay.block_tables.shape[1]
    tables = np.full((bucket, W), -1, np.int32)
    tables[:live] = lay.block_tables

    # fixed device buffers the graph is captured on
    kc, vc = dev(val.k_cache), dev(val.v_cache)
    q_d = torch.zeros((bucket, HQ, D), dtype=torch.bfloat16, device="cuda")
    kn_d = torch.zeros((bucket, HKV, D), dtype=torch.bfloat16, device="cuda")
    vn_d = torch.zeros_like(kn_d)
    slots_d = torch.full((bucket,), -1, dtype=torch.int64, device="cuda")
    tables_d = dev(tables)
    ctx_d = torch.zeros((bucket,), dtype=torch.int32, device="cuda")
    ws = pkv.decode_workspace(bucket, HQ, HKV, D, CAP, 0)
    out_d = torch.empty((bucket, HQ, D), dtype=torch.bfloat16, device="cuda")

    def step():
        pkv.kv_store(kn_d, vn_d, slots_d, kc, vc)
        pkv.paged_decode_attn(q_d, kc, vc, tables_d, ctx_d, CAP, lay.scale, workspace=ws,
                              out=out_d)

    step()                                   # first call on the device, outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()

    kc_h, vc_h = val.k_cache.copy(), val.v_cache.copy()
    for t in range(STEPS):
        ctx = np.zeros(bucket, np.int32)
        ctx[:live] = final - (STEPS - 1 - t)
        slots = _slots(tables, ctx)
        q = w.host_bf16_normal(g, (bucket, HQ, D))
        kn = w.host_bf16_normal(g, (bucket, HKV, D))
        vn = w.host_bf16_normal(g, (bucket, HKV, D))
        q_d.copy_(dev(q))
        kn_d.copy_(dev(kn))
        vn_d.copy_(dev(vn))
        slots_d.copy_(dev(slots))
        ctx_d.copy_(dev(ctx))
        graph.replay()
        torch.cuda.synchronize()
        got = out_d.clone()

        oracle.kv_store(kn, vn, slots, kc_h, vc_h)
        ref = oracle.paged_decode(q, kc_h, vc_h, tables, ctx, lay.scale)
        assert_attention_close(got, ref, f"bucket {bucket} step {t}")
        assert not host_bits(got)[live:].any(), "padding rows must be zero"
        # the pool after the graph's store equals the oracle's, bit for bit
        assert np.array_equal(host_bits(kc), kc_h) and np.array_equal(host_bits(vc), vc_h)

        # an eager call on the same buffers gives the same bits (the store rewrites the
        # same rows with the same values)
        step()
        torch.cuda.synchronize()
        assert torch.equal(out_d.view(torch.int16), got.view(torch.int16))
    assert pkv.get_device_errors() == 0
