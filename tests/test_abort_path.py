"""The abort path: once the device error word holds PKV_DEVERR_TIMEOUT (what a wait that gave
up leaves behind), every kernel of the library returns without computing or writing, and
after the word is cleared the same calls give correct results again.

The bit is raised from the host (pkv_raise_device_errors), so nothing here waits out a limit
or stalls the GPU. Decode is run in each launch shape it has: a static grid whose splits
merge in a thread-block cluster, a static grid with one split, a static grid whose splits
merge through global memory, and the work-queue grid.
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

SENTINEL = 0x7FC1  # a bf16 NaN that no kernel writes


def _filled_like(t: torch.Tensor) -> torch.Tensor:
    return torch.full(t.shape, SENTINEL, dtype=torch.int16, device=t.device).view(torch.bfloat16)


def _untouched(t: torch.Tensor) -> bool:
    return bool((t.view(torch.int16) == SENTINEL).all().item())


def _decode_case(ctx, seed):
    """A decode batch whose pools already hold the new token (stored by the oracle)."""
    g = w.rng(seed)
    lay = w.decode_layout(np.asarray(ctx, np.int32), w.blocks_needed(ctx) + 4, g)
    val = w.decode_values(lay, g)
    oracle.kv_store(val.k_new, val.v_new, lay.slot_mapping, val.k_cache, val.v_cache)
    return lay, val


# (contexts, num_splits): cluster merge, one split, global merge (9 splits), work queue
DECODE_SHAPES = [
    ([700, 1500, 64], 2),
    ([700, 1500, 64], 1),
    ([4000, 3000], 9),
    ([200] * 48, 1),  # 48 sequences x 8 KV heads = 384 units: more than two per SM
]


def _decode(lay, val, ns, out):
    return pkv.paged_decode_attn(dev(val.q), dev(val.k_cache), dev(val.v_cache),
                                 dev(lay.block_tables), dev(lay.context_lens),
                                 lay.max_context_len, lay.scale, num_splits=ns, out=out)


def test_abort_bit_stops_every_kernel_and_clearing_it_recovers():
    cases = [(_decode_case(ctx, 900 + i), ns) for i, (ctx, ns) in enumerate(DECODE_SHAPES)]
    # store inputs
    g = w.rng(950)
    lay_s, val_s = cases[0][0]
    kc_s, vc_s = dev(val_s.k_cache), dev(val_s.v_cache)
    # prefill inputs: two sequences, packed
    lens = np.array([100, 300], np.int64)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q_p = w.host_bf16_normal(g, (int(cu[-1]), 16, 128))
    k_p = w.host_bf16_normal(g, (int(cu[-1]), 8, 128))
    v_p = w.host_bf16_normal(g, (int(cu[-1]), 8, 128))

    assert pkv.get_device_errors(reset=True) == 0
    pkv.raise_device_errors(pkv.DEVERR_TIMEOUT)
    try:
        for (lay, val), ns in cases:
            out = _filled_like(dev(val.q))
            _decode(lay, val, ns, out)
            assert _untouched(out), f"decode with {ns} splits wrote while aborted"
        before_k, before_v = host_bits(kc_s), host_bits(vc_s)
        pkv.kv_store(dev(val_s.k_new), dev(val_s.v_new), dev(lay_s.slot_mapping), kc_s, vc_s)
        assert np.array_equal(host_bits(kc_s), before_k)
        assert np.array_equal(host_bits(vc_s), before_v)
        out_p = _filled_like(dev(q_p))
        pkv.varlen_prefill_attn(dev(q_p), dev(k_p), dev(v_p), dev(cu), dev(cu), 300, 300,
                                128 ** -0.5, out=out_p)
        assert _untouched(out_p), "prefill wrote while aborted"
        # QK-norm + RoPE + store: neither q nor the pools are written
        T = int(cu[-1])
        qkv = dev(w.host_bf16_normal(g, (T, (16 + 2 * 8) * 128)))
        ones = torch.ones(128, dtype=torch.bfloat16, device="cuda")
        table = torch.from_numpy(w.random_cos_sin_table(g, 512, 128)).cuda()
        pos = torch.arange(T, dtype=torch.int64, device="cuda") % 512
        slots = torch.arange(T, dtype=torch.int64, device="cuda")
        kc_r = _filled_like(torch.empty((-(-T // 256), 256, 8, 128), dtype=torch.bfloat16,
                                        device="cuda"))
        vc_r = _filled_like(kc_r)
        q_r = _filled_like(torch.empty((T, 16, 128), dtype=torch.bfloat16, device="cuda"))
        pkv.qk_norm_rope_store(qkv, pos, ones, ones, 1e-6, table, slots, kc_r, vc_r, 16, 8,
                               q_out=q_r)
        assert _untouched(q_r) and _untouched(kc_r) and _untouched(vc_r), \
            "qk_norm_rope_store wrote while aborted"
        assert pkv.get_device_errors(reset=False) == pkv.DEVERR_TIMEOUT
    finally:
        pkv.get_device_errors(reset=True)

    # cleared: the same calls compute again
    for (lay, val), ns in cases:
        out = _filled_like(dev(val.q))
        _decode(lay, val, ns, out)
        ref = oracle.paged_decode(val.q, val.k_cache, val.v_cache, lay.block_tables,
                                  lay.context_lens, lay.scale)
        assert_attention_close(out, ref, f"after clearing, {ns} splits")
    assert pkv.get_device_errors() == 0
