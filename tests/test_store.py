"""kv_store on the GPU against the oracle: bit-exact pools, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import workloads as w
from gpu_util import canary_pool, dev, host_bits
from libbuild import build_and_import

pytestmark = pytest.mark.gpu
pkv = build_and_import()


def _store_case(T, nb, bs, hkv, d, seed, neg=()):
    g = w.rng(seed)
    k = w.host_bf16_normal(g, (T, hkv, d))
    v = w.host_bf16_normal(g, (T, hkv, d))
    slots = g.permutation(nb * bs)[:T].astype(np.int64)
    for i in neg:
        slots[i] = -1
    kc = np.full((nb, bs, hkv, d), w.BF16_NAN_CANARY, np.uint16)
    return k, v, slots, kc


def _run_both(k, v, slots, kc_host, kd=None, vd=None):
    kc_o, vc_o = kc_host.copy(), kc_host.copy()
    oracle.kv_store(k, v, slots, kc_o, vc_o)
    kc_d, vc_d = dev(kc_host), dev(kc_host)
    pkv.kv_store(dev(k) if kd is None else kd, dev(v) if vd is None else vd, dev(slots), kc_d, vc_d)
    torch.cuda.synchronize()
    return kc_o, vc_o, host_bits(kc_d), host_bits(vc_d)


def test_store_tiny_decode_step():
    lay, val = w.tiny_decode()
    kc_o, vc_o = val.k_cache.copy(), val.v_cache.copy()
    oracle.kv_store(val.k_new, val.v_new, lay.slot_mapping, kc_o, vc_o)
    kc_d, vc_d = dev(val.k_cache), dev(val.v_cache)
    pkv.kv_store(dev(val.k_new), dev(val.v_new), dev(lay.slot_mapping), kc_d, vc_d)
    assert np.array_equal(host_bits(kc_d), kc_o)
    assert np.array_equal(host_bits(vc_d), vc_o)
    assert pkv.get_device_errors() == 0


@pytest.mark.parametrize("hkv,d,bs", [(8, 128, 16), (4, 128, 16), (16, 128, 16), (2, 64, 16),
                                      (3, 40, 16), (3, 4, 16), (64, 128, 4), (200, 128, 2)])
def test_store_row_shapes(hkv, d, bs):
    """Bulk copies through shared memory for rows that are whole 16-byte vectors (any count;
    16 KiB rows stage three tokens per CTA instead of eight);
    16-byte vectors straight through for rows too long to stage (200 x 128 bf16 = 50 KiB); a
    2-byte path for rows that are not whole vectors (3 x 4 bf16 = 24 bytes)."""
    k, v, slots, kc = _store_case(77, 6 if bs == 16 else 48, bs, hkv, d, 5, neg=(3, 40))
    assert len(slots) <= kc.shape[0] * kc.shape[1]
    kc_o, vc_o, kc_g, vc_g = _run_both(k, v, slots, kc)
    assert np.array_equal(kc_g, kc_o) and np.array_equal(vc_g, vc_o)


def test_store_strided_views_of_fused_qkv():
    g = w.rng(6)
    T, hq, hkv, d, nb, bs = 50, 16, 8, 128, 4, 256
    qkv = w.host_bf16_normal(g, (T, (hq + 2 * hkv) * d))
    k = qkv[:, hq * d:(hq + hkv) * d].reshape(T, hkv, d)
    v = qkv[:, (hq + hkv) * d:].reshape(T, hkv, d)
    slots = g.permutation(nb * bs)[:T].astype(np.int64)
    kc = np.zeros((nb, bs, hkv, d), np.uint16)
    qkv_d = dev(qkv)
    kd = qkv_d[:, hq * d:(hq + hkv) * d].view(T, hkv, d)
    vd = qkv_d[:, (hq + hkv) * d:].view(T, hkv, d)
    kc_o, vc_o, kc_g, vc_g = _run_both(k, v, slots, kc, kd, vd)
    assert np.array_equal(kc_g, kc_o) and np.array_equal(vc_g, vc_o)


def test_store_slot_out_of_range_is_skipped_and_flagged():
    k, v, slots, kc = _store_case(10, 2, 256, 8, 128, 7)
    slots[4] = 2 * 256 + 5
    pkv.get_device_errors(reset=True)
    kc_d, vc_d = dev(kc), dev(kc)
    pkv.kv_store(dev(k), dev(v), dev(slots), kc_d, vc_d)
    assert pkv.get_device_errors() & pkv.DEVERR_SLOT_RANGE
    ok = np.ones(10, bool)
    ok[4] = False
    kc_o, vc_o = kc.copy(), kc.copy()
    oracle.kv_store(k[ok], v[ok], slots[ok], kc_o, vc_o)
    assert np.array_equal(host_bits(kc_d), kc_o) and np.array_equal(host_bits(vc_d), vc_o)


def test_store_zero_tokens_is_a_no_op():
    kc = canary_pool(2, 256, 8, 128)
    before = host_bits(kc)
    e = torch.empty((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    pkv.kv_store(e, e, torch.empty(0, dtype=torch.int64, device="cuda"), kc, kc)
    assert np.array_equal(host_bits(kc), before)


def test_store_varlen_prefill_full_size():
    """The varlen prefill workload: 256 prompts, lengths U[100, 1024] (~143k tokens),
    stored through slot_mapping into 256-token blocks; the whole pool compared bit for bit."""
    lay = w.varlen_prefill_layout(num_blocks=w.blocks_needed(w.varlen_prefill_lengths()) + 32)
    T = int(lay.seqlens_q.sum())
    kd = w.device_bf16_normal((T, 8, 128), 301)
    vd = w.device_bf16_normal((T, 8, 128), 302)
    kc_d = canary_pool(lay.num_blocks, 256, 8, 128)
    vc_d = canary_pool(lay.num_blocks, 256, 8, 128)
    pkv.kv_store(kd, vd, dev(lay.slot_mapping), kc_d, vc_d)
    torch.cuda.synchronize()
    for src, pool_d in ((kd, kc_d), (vd, vc_d)):
        want = np.full((lay.num_blocks, 256, 8, 128), w.BF16_NAN_CANARY, np.uint16)
        src_h = host_bits(src)
        oracle.kv_store(src_h, src_h, lay.slot_mapping, want, want.copy())
        assert np.array_equal(host_bits(pool_d), want)
    assert pkv.get_device_errors() == 0
