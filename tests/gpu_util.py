"""Helpers for the GPU parity tests: move workload arrays to the device and back, build
full-size device pools, and compare a bf16 device result with the float64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import workloads as w

TOL_ABS = 1e-2
TOL_REL = 1e-2


def dev(a: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bits (host) -> torch.bfloat16 on cuda; int arrays keep their dtype."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f64(t: torch.Tensor) -> np.ndarray:
    return w.bf16_bits_to_f32(host_bits(t)).astype(np.float64)


def assert_attention_close(got: torch.Tensor, ref: np.ndarray, what: str = "") -> float:
    """max |got - ref| <= 1e-2 + 1e-2 |ref| element by element (bf16 in, fp32 accumulate)."""
    g = host_f64(got)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(ref).all(), f"{what}: non-finite reference (inputs read unset slots?)"
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref)
    bound = TOL_ABS + TOL_REL * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance; first at "
                             f"{tuple(idx)}: got {g[tuple(idx)]}, ref {ref[tuple(idx)]}")
    return float(err.max())


def canary_pool(num_blocks: int, block_size: int, hkv: int, d: int) -> torch.Tensor:
    t = torch.full((num_blocks, block_size, hkv, d), w.BF16_NAN_CANARY, dtype=torch.int16,
                   device="cuda")
    return t.view(torch.bfloat16)


def fill_sequences_on_device(lay, seed: int):
    """Full-size decode pools: every referenced block drawn N(0,1) on the device, then the
    slots past each sequence's context set back to the NaN canary (never read)."""
    bs, hkv, d = lay.block_size, lay.num_kv_heads, lay.head_dim
    kc = canary_pool(lay.num_blocks, bs, hkv, d)
    vc = canary_pool(lay.num_blocks, bs, hkv, d)
    ids = np.unique(lay.block_tables[lay.block_tables >= 0])
    idt = torch.from_numpy(ids.astype(np.int64)).cuda()
    kc[idt] = w.device_bf16_normal((len(ids), bs, hkv, d), seed)
    vc[idt] = w.device_bf16_normal((len(ids), bs, hkv, d), seed + 1)
    canary = torch.tensor(w.BF16_NAN_CANARY, dtype=torch.int16).view(torch.bfloat16).item()
    for b, c in enumerate(lay.context_lens):
        c = int(c)
        if c % bs:
            last = int(lay.block_tables[b, (c - 1) // bs])
            kc[last, c % bs:] = canary
            vc[last, c % bs:] = canary
    return kc, vc


def compact_for_oracle(kc: torch.Tensor, vc: torch.Tensor, tables: np.ndarray):
    """Copy the blocks the tables reference to the host as a compact pool, and renumber the
    tables to it (a block permutation, which leaves attention unchanged)."""
    ids = np.unique(tables[tables >= 0])
    remap = np.full(max(int(kc.shape[0]), 1), -1, np.int64)
    remap[ids] = np.arange(len(ids))
    idt = torch.from_numpy(ids.astype(np.int64)).cuda()
    k_h = host_bits(kc[idt])
    v_h = host_bits(vc[idt])
    t2 = np.where(tables >= 0, remap[np.maximum(tables, 0)], -1).astype(np.int32)
    return k_h, v_h, t2


def remap_slots(tables: np.ndarray, slots: np.ndarray, block_size: int) -> np.ndarray:
    """The slots of the blocks `tables` reference, renumbered as compact_for_oracle renumbers
    the blocks (negative slots stay negative)."""
    ids = np.unique(tables[tables >= 0])
    remap = np.full(int(ids.max()) + 1 if len(ids) else 1, -1, np.int64)
    remap[ids] = np.arange(len(ids))
    s = np.asarray(slots, np.int64)
    blk = np.maximum(s, 0) // block_size
    out = remap[np.minimum(blk, len(remap) - 1)] * block_size + np.maximum(s, 0) % block_size
    assert (out[s >= 0] >= 0).all(), "a slot outside the referenced blocks"
    return np.where(s >= 0, out, s).astype(np.int64)
