"""CPU oracle for the paged KV cache path (numpy front end over a plain C library).

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this package: only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of ``bench.py`` use
it. It shares no code with the CUDA library; both take their inputs from ``workloads``.

Arrays of bf16 values are passed as ``uint16`` bit patterns. Attention results come back as
float64 arrays; the store works in place on ``uint16`` pools.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

OK, BAD_SLOT, DUP_SLOT, BAD_BLOCK, BAD_ARG, NO_MEMORY, BAD_POSITION = range(7)
_ERRORS = {BAD_SLOT: "slot out of range", DUP_SLOT: "duplicate slot in one call",
           BAD_BLOCK: "block id out of range / table too narrow", BAD_ARG: "bad argument",
           NO_MEMORY: "out of host memory", BAD_POSITION: "position outside the cos/sin cache"}


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(_ERRORS.get(code, f"oracle status {code}"))
        self.code = code


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_D = ctypes.c_double


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the oracle library (building it first when missing). ``path`` loads another
    build of the same source (used by the tests that plant mistakes in a copy)."""
    lib = ctypes.CDLL(path or _build.build())
    lib.pkv_oracle_max_threads.restype = _I32
    lib.pkv_oracle_kv_store.restype = _I32
    lib.pkv_oracle_kv_store.argtypes = [_P, _I64, _P, _I64, _P, _I64, _P, _P, _I64, _I32, _I32]
    lib.pkv_oracle_paged_decode.restype = _I32
    lib.pkv_oracle_paged_decode.argtypes = [_P, _P, _P, _P, _I32, _P, _I32, _I32, _I32, _I32,
                                            _I32, _I64, _D, _P, _I32]
    lib.pkv_oracle_varlen_prefill.restype = _I32
    lib.pkv_oracle_varlen_prefill.argtypes = [_P, _I64, _P, _P, _I64, _P, _P, _I32, _P, _I32,
                                              _I32, _I64, _I32, _I32, _I32, _D, _I32, _P, _I32]
    lib.pkv_oracle_qk_norm_rope.restype = _I32
    lib.pkv_oracle_qk_norm_rope.argtypes = [_P, _I64, _I64, _P, _P, _P, _D, _P, _I64, _I32,
                                            _I32, _I32, _P, _P, _P, _P]
    return lib


_LIB: ctypes.CDLL | None = None


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        _LIB = load()
    return _LIB


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(_P)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads(L: ctypes.CDLL | None = None) -> int:
    return int((L or lib()).pkv_oracle_max_threads())


def kv_store(k, v, slot_mapping, k_cache, v_cache, *, L: ctypes.CDLL | None = None) -> None:
    """k_cache/v_cache [NB, bs, Hkv, D] (or [slots, Hkv, D]) uint16, updated in place."""
    L = L or lib()
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    k = np.asarray(k, np.uint16)
    v = np.asarray(v, np.uint16)
    Hkv, D = k_cache.shape[-2], k_cache.shape[-1]
    row = Hkv * D
    T = int(np.asarray(slot_mapping).shape[0])
    # token strides of (possibly strided) views; the rest of a row must be contiguous
    ks = k.strides[0] // 2 if T else row
    vs = v.strides[0] // 2 if T else row
    for a in (k, v):
        assert a.size == 0 or (a.strides[-1] == 2 and a.strides[-2] == D * 2), "rows must be dense"
    slots = _c(slot_mapping, np.int64)
    num_slots = k_cache.size // row
    rc = L.pkv_oracle_kv_store(k.ctypes.data_as(_P), ks, v.ctypes.data_as(_P), vs,
                               _ptr(slots), T, _ptr(k_cache), _ptr(v_cache), num_slots, Hkv, D)
    if rc:
        raise OracleError(rc)


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale: float, *,
                 num_threads: int = 0, L: ctypes.CDLL | None = None) -> np.ndarray:
    """q [B, Hq, D]; pools [NB, bs, Hkv, D]; block_tables [B, W]; context_lens [B]."""
    L = L or lib()
    q = _c(q, np.uint16)
    kc = _c(k_cache, np.uint16)
    vc = _c(v_cache, np.uint16)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = kc.shape
    assert D == D2 and bt.ndim == 2 and bt.shape[0] == B
    out = np.zeros((B, Hq, D), np.float64)
    rc = L.pkv_oracle_paged_decode(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(cl),
                                   B, Hq, Hkv, D, bs, NB, float(scale), _ptr(out), num_threads)
    if rc:
        raise OracleError(rc)
    return out


def varlen_prefill(q, k, v, cu_seqlens_q, cu_seqlens_k, scale: float, *, causal: bool = True,
                   block_table=None, num_threads: int = 0,
                   L: ctypes.CDLL | None = None) -> np.ndarray:
    """q [Tq, Hq, D]. Without block_table, k/v are packed [Tk, Hkv, D]; with it, k/v are the
    pools [NB, bs, Hkv, D]. Returns [Tq, Hq, D] float64."""
    L = L or lib()
    q = _c(q, np.uint16)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    cq = _c(cu_seqlens_q, np.int32)
    ck = _c(cu_seqlens_k, np.int32)
    Tq, Hq, D = q.shape
    Hkv = k.shape[-2]
    N = cq.shape[0] - 1
    if block_table is not None:
        bt = _c(block_table, np.int32)
        NB, bs = k.shape[0], k.shape[1]
        W = bt.shape[1]
    else:
        bt, NB, bs, W = None, 0, 0, 0
    out = np.zeros((Tq, Hq, D), np.float64)
    rc = L.pkv_oracle_varlen_prefill(_ptr(q), Hq * D, _ptr(k), _ptr(v), Hkv * D, _ptr(cq),
                                     _ptr(ck), N, _ptr(bt), W, bs, NB, Hq, Hkv, D, float(scale),
                                     int(bool(causal)), _ptr(out), num_threads)
    if rc:
        raise OracleError(rc)
    return out


def qk_norm_rope(qkv, positions, q_weight, k_weight, eps: float, cos_sin, num_q_heads: int,
                 num_kv_heads: int, *, L: ctypes.CDLL | None = None):
    """qkv [T, (Hq + 2 Hkv) * D] (or a strided view with dense rows) uint16 bf16 bits;
    positions [T]; weights [D] uint16; cos_sin [max_position, D] float32.
    Returns (q [T, Hq, D], k [T, Hkv, D], q_normed, k_normed), float64."""
    L = L or lib()
    qkv = np.asarray(qkv, np.uint16)
    T = qkv.shape[0]
    D = int(np.asarray(q_weight).shape[0])
    assert qkv.strides[-1] == 2
    ts = qkv.strides[0] // 2 if T else (num_q_heads + 2 * num_kv_heads) * D
    pos = _c(positions, np.int64)
    qw, kw = _c(q_weight, np.uint16), _c(k_weight, np.uint16)
    cs = _c(cos_sin, np.float32)
    q = np.zeros((T, num_q_heads, D)); k = np.zeros((T, num_kv_heads, D))
    qn = np.zeros_like(q); kn = np.zeros_like(k)
    rc = L.pkv_oracle_qk_norm_rope(qkv.ctypes.data_as(_P), ts, T, _ptr(pos), _ptr(qw), _ptr(kw),
                                   float(eps), _ptr(cs), cs.shape[0], num_q_heads, num_kv_heads,
                                   D, _ptr(q), _ptr(k), _ptr(qn), _ptr(kn))
    if rc:
        raise OracleError(rc)
    return q, k, qn, kn

