"""QK RMSNorm + RoPE fused into the store (pkv_qk_norm_rope_store) against the oracle.

Bound, from the arithmetic (bf16 has an 8-bit significand, so round-to-nearest has unit
roundoff u = 2^-8): the kernel rounds the normalised head n to bf16 (|error| <= u |n| per
element), rotates it in fp32 (|c|, |s| <= 1, so a pair's error is at most u (|n_i| +
|n_{i+h}|)), and rounds the result to bf16 (another <= u |y| <= u (|n_i| + |n_{i+h}|)); fp32
products and rsqrt add ~1e-6 relative. So every output element must satisfy
|gpu - oracle| <= 2^-7 (|n_i| + |n_{i+h}|) + 1e-6, with n the oracle's exact normalised values
of the element's pair. Value heads are copied: bit-exact. Pool rows that no slot names keep
their canary.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as w
from gpu_util import canary_pool, dev, host_bits, host_f64
from libbuild import build_and_import

pytestmark = pytest.mark.gpu
pkv = build_and_import()

D, BS = 128, 256
EPS = 1e-6


def _pair_bound(n):
    h = n.shape[-1] // 2
    s = np.abs(n[..., :h]) + np.abs(n[..., h:])
    return 2.0 ** -7 * np.concatenate([s, s], axis=-1) + 1e-6


def _close(got, ref, n, what):
    err = np.abs(got - ref)
    bound = _pair_bound(n)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} elements out of bound; first at "
                           f"{tuple(np.argwhere(bad)[0])}")


def _case(T, hq, hkv, seed, max_pos=4096, extra_cols=0, pad_every=0, nb=None):
    g = w.rng(seed)
    row = (hq + 2 * hkv) * D
    full = w.host_bf16_normal(g, (T, row + extra_cols))
    qkv = full[:, :row]                                     # a strided view when extra_cols
    qw = w.f32_to_bf16_bits(g.normal(1.0, 0.2, D).astype(np.float32))
    kw = w.f32_to_bf16_bits(g.normal(1.0, 0.2, D).astype(np.float32))
    table = w.random_cos_sin_table(g, max_pos, D)
    pos = g.integers(0, max_pos, T).astype(np.int64)
    nb = nb or (-(-T // BS) + 2)
    slots = g.permutation(nb * BS)[:T].astype(np.int64)
    if pad_every:
        slots[::pad_every] = -1
    return full, qkv, qw, kw, table, pos, slots, nb


def _run_gpu(full, qkv, qw, kw, table, pos, slots, nb, hq, hkv):
    full_d = dev(full)
    qkv_d = full_d[:, :qkv.shape[1]]
    kc, vc = canary_pool(nb, BS, hkv, D), canary_pool(nb, BS, hkv, D)
    q = pkv.qk_norm_rope_store(qkv_d, dev(pos), dev(qw), dev(kw), EPS,
                               torch.from_numpy(table).cuda(), dev(slots), kc, vc, hq, hkv)
    return q, kc, vc


def _check(full, qkv, qw, kw, table, pos, slots, nb, hq, hkv, q, kc, vc, what):
    qr, kr, qn, kn = oracle.qk_norm_rope(qkv, pos, qw, kw, EPS, table, hq, hkv)
    _close(host_f64(q), qr, qn, f"{what}: q")
    kcache, vcache = host_bits(kc).reshape(-1, hkv, D), host_bits(vc).reshape(-1, hkv, D)
    live = slots >= 0
    k_got = w.bf16_bits_to_f32(kcache[slots[live]]).astype(np.float64)
    _close(k_got, kr[live], kn[live], f"{what}: k")
    v_src = qkv.reshape(qkv.shape[0], hq + 2 * hkv, D)[:, hq + hkv:]
    assert np.array_equal(vcache[slots[live]], v_src[live]), f"{what}: v"
    untouched = np.ones(nb * BS, bool)
    untouched[slots[live]] = False
    assert (kcache[untouched] == w.BF16_NAN_CANARY).all() and \
        (vcache[untouched] == w.BF16_NAN_CANARY).all(), f"{what}: rows not named by a slot"


@pytest.mark.parametrize("T,hq,hkv", [(1, 16, 8), (5, 16, 8), (257, 16, 8), (64, 8, 8),
                                      (33, 32, 4), (11, 96, 16), (3, 400, 8)])
def test_qk_norm_rope_store_matches_oracle(T, hq, hkv):
    """Eight tokens per CTA for the usual head counts; 128 heads (32 KiB rows) stage three
    tokens per CTA, and 416 heads (104 KiB rows) one."""
    c = _case(T, hq, hkv, seed=T + hq)
    q, kc, vc = _run_gpu(*c, hq, hkv)
    _check(*c, hq, hkv, q, kc, vc, f"T={T} hq={hq} hkv={hkv}")
    assert pkv.get_device_errors() == 0


def test_fused_qkv_view_and_padding_slots():
    """Rows of a wider buffer (token stride > row), and padding tokens (slot -1) that still
    get their q."""
    c = _case(100, 16, 8, seed=5, extra_cols=256, pad_every=7)
    q, kc, vc = _run_gpu(*c, 16, 8)
    _check(*c, 16, 8, q, kc, vc, "view + padding")
    assert pkv.get_device_errors() == 0


def test_bad_position_is_flagged():
    full, qkv, qw, kw, table, pos, slots, nb = _case(10, 16, 8, seed=6, max_pos=64)
    pos = pos.copy()
    pos[3] = 64                                              # one past the table
    pkv.get_device_errors(reset=True)
    q, kc, vc = _run_gpu(full, qkv, qw, kw, table, pos, slots, nb, 16, 8)
    assert pkv.get_device_errors() & pkv.DEVERR_POSITION_RANGE
    pkv.get_device_errors(reset=True)
    ok = np.arange(10) != 3
    qr, kr, qn, kn = oracle.qk_norm_rope(qkv[ok], pos[ok], qw, kw, EPS, table, 16, 8)
    _close(host_f64(q)[ok], qr, qn, "other tokens")


def test_full_varlen_prefill_tokens_sampled():
    """The varlen prefill workload's 145k new tokens (positions within their prompts, slots of
    the workload's block draw), every 101st token checked against the oracle; V and the
    untouched rows checked in full."""
    lens = w.varlen_prefill_lengths()
    lay = w.varlen_prefill_layout(num_blocks=w.blocks_needed(lens) + 64)
    T = int(lens.sum())
    g = w.rng(8)
    hq, hkv = 16, 8
    qkv_d = w.device_bf16_normal((T, (hq + 2 * hkv) * D), 801)
    qw = w.f32_to_bf16_bits(g.normal(1.0, 0.2, D).astype(np.float32))
    kw = w.f32_to_bf16_bits(g.normal(1.0, 0.2, D).astype(np.float32))
    table = w.random_cos_sin_table(g, 1024, D)
    pos = np.concatenate([np.arange(L) for L in lens]).astype(np.int64)
    slots = lay.slot_mapping
    kc, vc = canary_pool(lay.num_blocks, BS, hkv, D), canary_pool(lay.num_blocks, BS, hkv, D)
    q = pkv.qk_norm_rope_store(qkv_d, dev(pos), dev(qw), dev(kw), EPS,
                               torch.from_numpy(table).cuda(), dev(slots), kc, vc, hq, hkv)
    idx = np.arange(0, T, 101)
    qkv_s = host_bits(qkv_d[torch.from_numpy(idx).cuda()])
    qr, kr, qn, kn = oracle.qk_norm_rope(qkv_s, pos[idx], qw, kw, EPS, table, hq, hkv)
    _close(host_f64(q[torch.from_numpy(idx).cuda()]), qr, qn, "q (sampled)")
    kcache = host_bits(kc).reshape(-1, hkv, D)
    _close(w.bf16_bits_to_f32(kcache[slots[idx]]).astype(np.float64), kr, kn, "k (sampled)")
    vcache = host_bits(vc).reshape(-1, hkv, D)
    v_all = host_bits(qkv_d).reshape(T, hq + 2 * hkv, D)[:, hq + hkv:]
    assert np.array_equal(vcache[slots], v_all)
    assert pkv.get_device_errors() == 0
