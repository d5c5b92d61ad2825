"""Pins that tie the CPU oracle to something other than itself.

Each ``pin_*`` takes a loaded oracle library and raises ``AssertionError`` when the oracle
disagrees with what the nano-vLLM pages and the mathematics fix:

* library routines the paged operations reduce to: with the pages fixed to one physical
  layout, paged decode and varlen prefill are ordinary (GQA, causal) scaled-dot-product
  attention, which torch's CPU ``scaled_dot_product_attention`` computes in float64;
* closed forms: a one-token context returns that token's V; a zero query returns the mean
  of V; one key whose score dominates returns that key's V; the store is a row copy;
* invariants: permuting physical block ids leaves every output bit-identical; a shared,
  ref-counted prefix block gives the same result as a private copy; prefix-cached prefill
  gives the rows of the uncached computation (prefix caching computes only the remaining
  tokens: «企业官网建设流程全解析 (Nano-vLLM 指南)» §4.4); decode equals the last row of
  causal prefill over the same sequence.

``tests/test_oracle.py`` runs every pin on the oracle; ``tests/test_oracle_mutants.py`` plants
plausible mistakes in copies of the oracle's source and checks that some pin fails for each.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F

import oracle
import workloads as w


def _f64(bits: np.ndarray) -> np.ndarray:
    return w.bf16_bits_to_f32(bits).astype(np.float64)


def _sdpa(q, k, v, scale, causal=False):
    """q [Hq, Lq, D], k/v [Hkv, Lk, D] float64 -> [Hq, Lq, D] via torch's library routine."""
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(a)) for a in (q, k, v))
    return F.scaled_dot_product_attention(tq[None], tk[None], tv[None], scale=scale,
                                          is_causal=causal, enable_gqa=True)[0].numpy()


def _decode_case(ctx, bs, seed, hq=4, hkv=2, d=16, spare_blocks=3):
    g = w.rng(seed)
    nb = w.blocks_needed(ctx, bs) + spare_blocks
    lay = w.decode_layout(ctx, nb, g, block_size=bs, num_q_heads=hq, num_kv_heads=hkv, head_dim=d)
    val = w.decode_values(lay, g)
    kc, vc = val.k_cache.copy(), val.v_cache.copy()
    oracle.kv_store(val.k_new, val.v_new, lay.slot_mapping, kc, vc, L=_L)
    return lay, val, kc, vc


_L = None  # the library under test, set by run_pin


def _decode(L, lay, q, kc, vc, bt=None, ctx=None, scale=None):
    return oracle.paged_decode(q, kc, vc, lay.block_tables if bt is None else bt,
                               lay.context_lens if ctx is None else ctx,
                               lay.scale if scale is None else scale, L=L)


# ---------------------------------------------------------------------------------- store
def pin_store_is_row_copy(L):
    g = w.rng(11)
    nb, bs, hkv, d = 6, 4, 2, 8
    T = 9
    k = w.host_bf16_normal(g, (T, hkv, d))
    v = w.host_bf16_normal(g, (T, hkv, d))
    slots = g.permutation(nb * bs)[:T].astype(np.int64)
    slots[3] = -1                                  # a padding token: not stored
    kc = np.full((nb, bs, hkv, d), w.BF16_NAN_CANARY, np.uint16)
    vc = kc.copy()
    oracle.kv_store(k, v, slots, kc, vc, L=L)
    want_k = np.full((nb * bs, hkv, d), w.BF16_NAN_CANARY, np.uint16)
    want_v = want_k.copy()
    keep = slots >= 0
    want_k[slots[keep]] = k[keep]                  # numpy fancy-index scatter
    want_v[slots[keep]] = v[keep]
    assert np.array_equal(kc.reshape(nb * bs, hkv, d), want_k)
    assert np.array_equal(vc.reshape(nb * bs, hkv, d), want_v)
    # gathering back through slot_mapping returns the input
    assert np.array_equal(kc.reshape(nb * bs, hkv, d)[slots[keep]], k[keep])


def pin_store_strided_views(L):
    """k and v as views into one fused [T, (Hq + 2 Hkv) * D] qkv buffer."""
    g = w.rng(12)
    nb, bs, hq, hkv, d, T = 4, 4, 4, 2, 8, 7
    qkv = w.host_bf16_normal(g, (T, (hq + 2 * hkv) * d))
    k = qkv[:, hq * d:(hq + hkv) * d].reshape(T, hkv, d)
    v = qkv[:, (hq + hkv) * d:].reshape(T, hkv, d)
    slots = g.permutation(nb * bs)[:T].astype(np.int64)
    kc = np.zeros((nb, bs, hkv, d), np.uint16)
    vc = np.zeros_like(kc)
    oracle.kv_store(k, v, slots, kc, vc, L=L)
    assert np.array_equal(kc.reshape(-1, hkv, d)[slots], k)
    assert np.array_equal(vc.reshape(-1, hkv, d)[slots], v)


def pin_store_rejects_bad_slots(L):
    kc = np.zeros((2, 4, 1, 8), np.uint16)
    vc = kc.copy()
    k = np.ones((2, 1, 8), np.uint16)
    for slots, code in (([0, 8], oracle.BAD_SLOT), ([3, 3], oracle.DUP_SLOT)):
        try:
            oracle.kv_store(k, k, np.array(slots, np.int64), kc, vc, L=L)
        except oracle.OracleError as e:
            assert e.code == code
        else:
            raise AssertionError(f"slots {slots} accepted")


# --------------------------------------------------------------------------------- decode
def pin_decode_matches_sdpa(L):
    """Gathered through a random block table, each sequence's decode is plain GQA attention
    of its one query over its logical K/V."""
    for bs, ctx, seed in ((4, [1, 3, 4, 5, 13], 21), (16, [16, 40, 1, 33], 22),
                          (256, [1, 17, 255, 300], 1)):
        hq, hkv, d = (16, 8, 128) if bs == 256 else (4, 2, 16)
        lay, val, kc, vc = _decode_case(ctx, bs, seed, hq=hq, hkv=hkv, d=d)
        out = _decode(L, lay, val.q, kc, vc)
        for b, c in enumerate(ctx):
            want = _sdpa(_f64(val.q[b])[:, None, :],
                         _f64(val.logical_k[b]).transpose(1, 0, 2),
                         _f64(val.logical_v[b]).transpose(1, 0, 2), lay.scale)[:, 0, :]
            np.testing.assert_allclose(out[b], want, rtol=1e-12, atol=1e-12)


def pin_decode_scale_is_an_argument(L):
    lay, val, kc, vc = _decode_case([9, 14], 4, 23)
    for scale in (0.05, 0.7):
        out = _decode(L, lay, val.q, kc, vc, scale=scale)
        for b in range(2):
            want = _sdpa(_f64(val.q[b])[:, None, :], _f64(val.logical_k[b]).transpose(1, 0, 2),
                         _f64(val.logical_v[b]).transpose(1, 0, 2), scale)[:, 0, :]
            np.testing.assert_allclose(out[b], want, rtol=1e-12, atol=1e-12)


def pin_decode_context_one_returns_v(L):
    lay, val, kc, vc = _decode_case([1, 1, 1], 4, 24)
    out = _decode(L, lay, val.q, kc, vc)
    group = lay.num_q_heads // lay.num_kv_heads
    for b in range(3):
        v0 = _f64(val.logical_v[b][0])            # [Hkv, D]
        assert np.array_equal(out[b], np.repeat(v0, group, axis=0))


def pin_decode_zero_query_is_mean_of_v(L):
    lay, val, kc, vc = _decode_case([7, 12], 4, 25)
    q0 = np.zeros_like(val.q)
    out = _decode(L, lay, q0, kc, vc)
    group = lay.num_q_heads // lay.num_kv_heads
    for b in range(2):
        mean = _f64(val.logical_v[b]).mean(axis=0)  # [Hkv, D]
        np.testing.assert_allclose(out[b], np.repeat(mean, group, axis=0), rtol=1e-13, atol=1e-13)


def pin_decode_dominant_key(L):
    """q = 64 * k_j: the score of key j exceeds every other by hundreds, so the output is v_j
    (to far below bf16 resolution). The scores overflow exp() unless the maximum is taken out."""
    lay, val, kc, vc = _decode_case([11], 4, 26)
    j = 6
    group = lay.num_q_heads // lay.num_kv_heads
    kj = w.bf16_bits_to_f32(val.logical_k[0][j])                     # [Hkv, D]
    q = w.f32_to_bf16_bits(64.0 * np.repeat(kj, group, axis=0))[None]
    out = _decode(L, lay, q, kc, vc)
    want = np.repeat(_f64(val.logical_v[0][j]), group, axis=0)
    np.testing.assert_allclose(out[0], want, rtol=0, atol=1e-6)


def pin_decode_block_permutation_invariant(L):
    lay, val, kc, vc = _decode_case([5, 13, 2, 9], 4, 27, spare_blocks=5)
    base = _decode(L, lay, val.q, kc, vc)
    perm = w.rng(99).permutation(lay.num_blocks)    # new id of old block b is perm[b]
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = np.where(lay.block_tables >= 0, perm[np.maximum(lay.block_tables, 0)], -1)
    moved = _decode(L, lay, val.q, kc2, vc2, bt=bt2.astype(np.int32))
    assert np.array_equal(base, moved)


def pin_decode_gqa_equals_mha_on_replicated_heads(L):
    lay, val, kc, vc = _decode_case([6, 10], 4, 28)
    group = lay.num_q_heads // lay.num_kv_heads
    gqa = _decode(L, lay, val.q, kc, vc)
    kc_m = np.ascontiguousarray(np.repeat(kc, group, axis=2))
    vc_m = np.ascontiguousarray(np.repeat(vc, group, axis=2))
    mha = _decode(L, lay, val.q, kc_m, vc_m)
    assert np.array_equal(gqa, mha)


def pin_decode_empty_context_is_zero(L):
    lay, val, kc, vc = _decode_case([3, 5], 4, 29)
    ctx = lay.context_lens.copy()
    ctx[1] = 0
    out = _decode(L, lay, val.q, kc, vc, ctx=ctx)
    assert np.array_equal(out[1], np.zeros_like(out[1]))


# -------------------------------------------------------------------------------- prefill
def _prefill_case(lens, seed, bs=4, hq=4, hkv=2, d=16):
    g = w.rng(seed)
    lay = w.prefill_layout(lens, w.blocks_needed(lens, bs) + 2, g, block_size=bs)
    lay.num_q_heads, lay.num_kv_heads, lay.head_dim = hq, hkv, d
    val = w.prefill_values(lay, g)
    return lay, val


def pin_prefill_matches_sdpa(L):
    lens = [1, 5, 8, 13]
    lay, val = _prefill_case(lens, 31)
    cq = lay.cu_seqlens_q
    for causal in (True, False):
        out = oracle.varlen_prefill(val.q, val.k, val.v, cq, cq, lay.scale, causal=causal, L=L)
        for n in range(len(lens)):
            a, b = cq[n], cq[n + 1]
            want = _sdpa(_f64(val.q[a:b]).transpose(1, 0, 2), _f64(val.k[a:b]).transpose(1, 0, 2),
                         _f64(val.v[a:b]).transpose(1, 0, 2), lay.scale, causal=causal)
            np.testing.assert_allclose(out[a:b], want.transpose(1, 0, 2), rtol=1e-12, atol=1e-12)


def pin_prefill_paged_equals_packed(L):
    lens = [3, 9, 4]
    lay, val = _prefill_case(lens, 32)
    cq = lay.cu_seqlens_q
    kc, vc = val.k_cache.copy(), val.v_cache.copy()
    oracle.kv_store(val.k, val.v, lay.slot_mapping, kc, vc, L=L)
    packed = oracle.varlen_prefill(val.q, val.k, val.v, cq, cq, lay.scale, L=L)
    paged = oracle.varlen_prefill(val.q, kc, vc, cq, cq, lay.scale, block_table=lay.block_table, L=L)
    assert np.array_equal(packed, paged)


def _prefix_case(suffix, prefix_len, seed, private=False, bs=4):
    g = w.rng(seed)
    nb = 64
    lay = w.prefix_prefill_layout(suffix, prefix_len, nb, g, block_size=bs, private_prefix=private)
    lay.num_q_heads, lay.num_kv_heads, lay.head_dim = 4, 2, 16
    val = w.prefill_values(lay, w.rng(seed + 1000))
    kc, vc = val.k_cache.copy(), val.v_cache.copy()
    rows = w.suffix_rows(lay)
    oracle.kv_store(val.k[rows], val.v[rows], lay.slot_mapping, kc, vc, L=_L)
    return lay, val, kc, vc


def pin_prefix_cache_gives_uncached_rows(L):
    """Queries over the suffix only, keys through block_table (prefix + suffix), equal the
    suffix rows of causal prefill over whole sequences."""
    suffix, P = [3, 6, 1], 8
    lay, val, kc, vc = _prefix_case(suffix, P, 41)
    cached = oracle.varlen_prefill(val.q, kc, vc, lay.cu_seqlens_q, lay.cu_seqlens_k, lay.scale,
                                   block_table=lay.block_table, L=L)
    # uncached: every token of every sequence is a query; pad q with fresh rows for the prefix
    ck = lay.cu_seqlens_k
    rows = w.suffix_rows(lay)
    q_full = np.zeros((int(ck[-1]),) + val.q.shape[1:], np.uint16)
    q_full[rows] = val.q
    full = oracle.varlen_prefill(q_full, val.k, val.v, ck, ck, lay.scale, L=L)
    assert np.array_equal(cached, full[rows])


def pin_shared_prefix_equals_private_copy(L):
    suffix, P = [5, 2, 7], 8
    shared = _prefix_case(suffix, P, 42)
    private = _prefix_case(suffix, P, 42, private=True)
    assert (shared[0].ref_count.max() == len(suffix) and private[0].ref_count.max() == 1)
    outs = []
    for lay, val, kc, vc in (shared, private):
        outs.append(oracle.varlen_prefill(val.q, kc, vc, lay.cu_seqlens_q, lay.cu_seqlens_k,
                                          lay.scale, block_table=lay.block_table, L=L))
    assert np.array_equal(outs[0], outs[1])


def pin_decode_is_last_prefill_row(L):
    lens = [6, 11]
    lay, val = _prefill_case(lens, 43)
    cq = lay.cu_seqlens_q
    kc, vc = val.k_cache.copy(), val.v_cache.copy()
    oracle.kv_store(val.k, val.v, lay.slot_mapping, kc, vc, L=L)
    pre = oracle.varlen_prefill(val.q, val.k, val.v, cq, cq, lay.scale, L=L)
    last = cq[1:] - 1
    dec = oracle.paged_decode(val.q[last], kc, vc, lay.block_table, np.array(lens, np.int32),
                              lay.scale, L=L)
    assert np.array_equal(dec, pre[last])


def pin_prefill_rows_without_keys_are_zero(L):
    """Causal with more queries than keys: the first Lq - Lk queries see no key."""
    g = w.rng(44)
    q = w.host_bf16_normal(g, (5, 4, 16))
    k = w.host_bf16_normal(g, (2, 2, 16))
    v = w.host_bf16_normal(g, (2, 2, 16))
    out = oracle.varlen_prefill(q, k, v, np.array([0, 5], np.int32), np.array([0, 2], np.int32),
                                0.25, L=L)
    assert np.array_equal(out[:3], np.zeros_like(out[:3]))
    want = _sdpa(_f64(q[3:]).transpose(1, 0, 2), _f64(k).transpose(1, 0, 2),
                 _f64(v).transpose(1, 0, 2), 0.25, causal=True)
    np.testing.assert_allclose(out[3:], want.transpose(1, 0, 2), rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------- QK normalisation + RoPE
def _qkv_case(T, hq, hkv, d, seed):
    g = w.rng(seed)
    return w.host_bf16_normal(g, (T, (hq + 2 * hkv) * d)), g


def _table(angles: np.ndarray) -> np.ndarray:
    """cos/sin table rows [cos(a_0..a_{h-1}), sin(a_0..a_{h-1})] as float32."""
    return np.concatenate([np.cos(angles), np.sin(angles)], axis=-1).astype(np.float32)


ONE = 0x3F80  # bf16 1.0


def pin_qknorm_unit_rms_and_direction(L):
    """Weight 1, eps 0, no rotation: every head comes out with RMS exactly 1, in the direction
    of its input."""
    d, hq, hkv = 16, 3, 2
    qkv, _ = _qkv_case(5, hq, hkv, d, 1)
    one = np.full(d, ONE, np.uint16)
    q, k, qn, kn = oracle.qk_norm_rope(qkv, np.zeros(5), one, one, 0.0, _table(np.zeros((1, d // 2))),
                                       hq, hkv, L=L)
    np.testing.assert_allclose(q, qn, rtol=0, atol=0)
    x = _f64(qkv).reshape(5, hq + 2 * hkv, d)
    for y, xs in ((qn, x[:, :hq]), (kn, x[:, hq:hq + hkv])):
        np.testing.assert_allclose(np.sqrt((y ** 2).mean(-1)), 1.0, rtol=1e-12)
        cosang = (y * xs).sum(-1) / np.linalg.norm(y, axis=-1) / np.linalg.norm(xs, axis=-1)
        np.testing.assert_allclose(cosang, 1.0, rtol=1e-12)


def pin_qknorm_eps_closed_form(L):
    """A constant head of value c with eps: each element becomes c / sqrt(c^2 + eps)."""
    d = 8
    qkv = np.full((1, 3 * d), ONE, np.uint16)                    # all ones, hq = hkv = 1
    one = np.full(d, ONE, np.uint16)
    _, _, qn, kn = oracle.qk_norm_rope(qkv, [0], one, one, 0.5, _table(np.zeros((1, d // 2))),
                                       1, 1, L=L)
    np.testing.assert_allclose(qn, 1 / np.sqrt(1.5), rtol=1e-14)
    np.testing.assert_allclose(kn, 1 / np.sqrt(1.5), rtol=1e-14)


def pin_qknorm_weight_is_elementwise(L):
    d, hq, hkv = 16, 2, 1
    qkv, g = _qkv_case(3, hq, hkv, d, 2)
    one = np.full(d, ONE, np.uint16)
    wq, wk = w.host_bf16_normal(g, (d,)), w.host_bf16_normal(g, (d,))
    t = _table(np.zeros((1, d // 2)))
    _, _, qn1, kn1 = oracle.qk_norm_rope(qkv, np.zeros(3), one, one, 1e-6, t, hq, hkv, L=L)
    _, _, qn, kn = oracle.qk_norm_rope(qkv, np.zeros(3), wq, wk, 1e-6, t, hq, hkv, L=L)
    np.testing.assert_allclose(qn, qn1 * _f64(wq), rtol=1e-14)
    np.testing.assert_allclose(kn, kn1 * _f64(wk), rtol=1e-14)


def pin_rope_rotates_i_with_i_plus_half(L):
    """A head that is the unit vector e_i (normalised to sqrt(d) e_i) at angle a_i: element i
    becomes sqrt(d) cos a_i and element i + d/2 becomes sqrt(d) sin a_i (and e_{i+d/2} gives
    -sqrt(d) sin a_i and sqrt(d) cos a_i); nothing else changes."""
    d, half = 8, 4
    angles = np.array([[0.3, -1.1, 2.0, 0.7]])
    one = np.full(d, ONE, np.uint16)
    for i in range(d):
        qkv = np.zeros((1, 3 * d), np.uint16)
        qkv[0, i] = ONE
        qkv[0, d + i] = ONE
        q, k, _, _ = oracle.qk_norm_rope(qkv, [0], one, one, 0.0, _table(angles), 1, 1, L=L)
        t = _table(angles).astype(np.float64)[0]
        c, s = t[i % half], t[half + i % half]
        want = np.zeros(d)
        if i < half:
            want[i], want[i + half] = c, s
        else:
            want[i - half], want[i] = -s, c
        want *= np.sqrt(d)
        np.testing.assert_allclose(q[0, 0], want, atol=1e-12)
        np.testing.assert_allclose(k[0, 0], want, atol=1e-12)


def pin_rope_relative_position(L):
    """With the standard table (angle p * 10000^(-2i/d)), the score between a rotated query at
    position m and key at n depends on m - n only."""
    d, hq, hkv = 32, 1, 1
    P = 64
    inv = 10000.0 ** (-np.arange(0, d, 2) / d)
    table = _table(np.arange(P)[:, None] * inv[None, :])
    qkv, _ = _qkv_case(1, hq, hkv, d, 3)
    one = np.full(d, ONE, np.uint16)
    rows = np.repeat(qkv, 4, axis=0)
    q, k, _, _ = oracle.qk_norm_rope(rows, [5, 20, 2, 17], one, one, 1e-6, table, hq, hkv, L=L)
    # (m, n) = (5, 2) and (20, 17): the same distance
    np.testing.assert_allclose((q[0, 0] * k[2, 0]).sum(), (q[1, 0] * k[3, 0]).sum(), rtol=1e-5)


def pin_rope_keeps_pair_norms(L):
    d, hq, hkv = 16, 2, 2
    qkv, g = _qkv_case(4, hq, hkv, d, 4)
    one = np.full(d, ONE, np.uint16)
    table = _table(g.uniform(-np.pi, np.pi, (7, d // 2)))
    q, k, qn, kn = oracle.qk_norm_rope(qkv, [0, 6, 3, 3], one, one, 1e-6, table, hq, hkv, L=L)
    for y, n in ((q, qn), (k, kn)):
        h = d // 2
        np.testing.assert_allclose(y[..., :h] ** 2 + y[..., h:] ** 2,
                                   n[..., :h] ** 2 + n[..., h:] ** 2, rtol=1e-6)


def pin_qknorm_rejects_bad_position(L):
    qkv, _ = _qkv_case(2, 1, 1, 8, 5)
    one = np.full(8, ONE, np.uint16)
    try:
        oracle.qk_norm_rope(qkv, [0, 4], one, one, 0.0, _table(np.zeros((4, 4))), 1, 1, L=L)
    except oracle.OracleError as e:
        assert e.code == oracle.BAD_POSITION
    else:
        raise AssertionError("position 4 of a 4-row table was accepted")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


def run_pin(pin, L):
    global _L
    _L = L
    try:
        pin(L)
    finally:
        _L = None
