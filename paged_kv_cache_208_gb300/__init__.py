"""Paged KV cache kernels for GB300 (sm_103a): a thin Python binding over libpkv's C ABI.

The functions here only marshal arguments: they check dtype, device and layout of torch
tensors, pass raw device pointers and the current CUDA stream to the ``pkv_*`` entry points
declared in ``include/pkv.h``, and raise ``PkvError`` on a non-zero status. Every step of
the computation runs in the CUDA library; there is no other implementation to fall back
to. Importing this package fails if ``libpkv.so`` has not been built
(``python paged_kv_cache_208_gb300/build.py`` or ``__graft_entry__.build()``).

PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_NO_BLOCKS = range(6)
DEVERR_SLOT_RANGE, DEVERR_BLOCK_RANGE, DEVERR_CONTEXT_RANGE = 1, 2, 4
DEVERR_SEQLEN_RANGE, DEVERR_TIMEOUT, DEVERR_POSITION_RANGE = 8, 16, 32
DEVERR_WORKSPACE = 64

# symbol -> (restype, argtypes); mirrors include/pkv.h
_P, _I32, _I64, _F, _SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                           ctypes.c_size_t)
SIGNATURES = {
    "pkv_status_string": (ctypes.c_char_p, [_I32]),
    "pkv_abi_version": (_I32, []),
    "pkv_get_device_errors": (_I32, [ctypes.POINTER(ctypes.c_uint32), _I32]),
    "pkv_raise_device_errors": (_I32, [ctypes.c_uint32]),
    "pkv_kv_store": (_I32, [_P, _I64, _P, _I64, _P, _I64, _P, _P, _I64, _I32, _I32, _P]),
    "pkv_decode_workspace_bytes": (_SZ, [_I32, _I32, _I32, _I32, _I32, _I32]),
    "pkv_paged_decode_attn": (_I32, [_P, _P, _P, _P, _I32, _P, _I32, _I32, _I32, _I32, _I32,
                                     _I32, _I64, _F, _I32, _P, _SZ, _P, _P]),
    "pkv_paged_decode_attn_noalloc": (_I32, [_P, _P, _P, _P, _I32, _P, _I32, _I32, _I32, _I32,
                                             _I32, _I32, _I64, _F, _I32, _P, _P]),
    "pkv_paged_decode_step": (_I32, [_P, _P, _I64, _P, _I64, _P, _P, _P, _P, _I32, _P, _I32,
                                     _I32, _I32, _I32, _I32, _I32, _I64, _F, _I32, _P, _SZ,
                                     _P, _P]),
    "pkv_prefill_workspace_bytes": (_SZ, [_I32, _I32, _I32, _I32]),
    "pkv_varlen_prefill_attn": (_I32, [_P, _I64, _I64, _P, _P, _I64, _I64, _P, _P, _I32, _I32,
                                       _I32, _P, _I32, _I32, _I64, _I32, _I32, _I32, _F, _I32,
                                       _P, _SZ, _P, _P]),
    "pkv_qk_norm_rope_store": (_I32, [_P, _I64, _I64, _P, _P, _P, _F, _P, _I64, _P, _P, _P,
                                      _P, _I64, _I32, _I32, _I32, _P]),
    "pkv_bm_create": (_P, [_I32, _I32]),
    "pkv_bm_destroy": (None, [_P]),
    "pkv_bm_num_free": (_I32, [_P]),
    "pkv_bm_ref_count": (_I32, [_P, _I32]),
    "pkv_bm_block_hash": (_I32, [_P, _I32, ctypes.POINTER(ctypes.c_uint64),
                                 ctypes.POINTER(ctypes.c_int32)]),
    "pkv_bm_allocate": (_I32, [_P, _P, _I32, _P, _I32, ctypes.POINTER(ctypes.c_int32),
                               ctypes.POINTER(ctypes.c_int32)]),
    "pkv_bm_deallocate": (_I32, [_P, _P, _I32]),
    "pkv_bm_can_append": (_I32, [_P, _I32]),
    "pkv_bm_may_append": (_I32, [_P, _P, _I32, _P, _I32, ctypes.POINTER(ctypes.c_int32)]),
    "pkv_xxh64": (ctypes.c_uint64, [_P, _SZ, ctypes.c_uint64]),
}


class PkvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {_LIB.pkv_status_string(status).decode()} (status {status})")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          f"`python {os.path.join(_HERE, 'build.py')}` (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_LIB = _load()


def lib() -> ctypes.CDLL:
    """The loaded C library (for callers that want the raw C ABI)."""
    return _LIB


def _check(fn: str, status: int) -> None:
    if status != OK:
        raise PkvError(fn, status)


# The current stream's cudaStream_t for a device index, without building a Stream object
# (several microseconds a call); the public query when this torch lacks it.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int:
    if stream is None:
        if _raw_stream is not None:
            return int(_raw_stream(torch.cuda.current_device()))
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream if hasattr(stream, "cuda_stream") else stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype: torch.dtype) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def get_device_errors(reset: bool = True) -> int:
    """OR of the PKV_DEVERR_* bits kernels set since the last reset (synchronises)."""
    v = ctypes.c_uint32(0)
    _check("pkv_get_device_errors", _LIB.pkv_get_device_errors(ctypes.byref(v), int(reset)))
    return int(v.value)


def raise_device_errors(bits: int) -> None:
    """OR PKV_DEVERR_* bits into the device error word (synchronises). DEVERR_TIMEOUT makes
    every later kernel return without computing until get_device_errors(reset=True)."""
    _check("pkv_raise_device_errors", _LIB.pkv_raise_device_errors(int(bits)))


def kv_store(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
             k_cache: torch.Tensor, v_cache: torch.Tensor, stream=None) -> None:
    """k_cache[slot_mapping[t]] = k[t]; v_cache[slot_mapping[t]] = v[t] (negative slot = skip).

    k, v: [T, Hkv, D] bf16 with dense rows (token stride may be larger, e.g. views into a
    fused qkv tensor); slot_mapping: [T] int64; caches: [NB, bs, Hkv, D] bf16, contiguous.
    """
    for t, n in ((k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.bfloat16)
    _need(slot_mapping, "slot_mapping", torch.int64)
    hkv, d = k_cache.shape[-2], k_cache.shape[-1]
    for t, n in ((k, "k"), (v, "v")):
        if t.dim() != 3 or t.shape[1:] != (hkv, d) or t.stride(2) != 1 or t.stride(1) != d:
            raise ValueError(f"{n} must be [T, {hkv}, {d}] with dense rows")
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("caches must be contiguous")
    T = slot_mapping.shape[0]
    _check("pkv_kv_store", _LIB.pkv_kv_store(
        _ptr(k), k.stride(0) if T else hkv * d, _ptr(v), v.stride(0) if T else hkv * d,
        _ptr(slot_mapping.contiguous()), T, _ptr(k_cache), _ptr(v_cache),
        k_cache.numel() // (hkv * d), hkv, d, _stream(stream)))


def decode_workspace_bytes(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                           max_context_len: int, num_splits: int = 0) -> int:
    return int(_LIB.pkv_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim,
                                               max_context_len, num_splits))


def decode_workspace(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                     max_context_len: int, num_splits: int = 0, device=None,
                     stream=None) -> torch.Tensor:
    """A decode workspace, zeroed on `stream` (the current stream when None): its first word
    is the split kernel's work counter, which must be zero before the first call (every call
    leaves it at zero again). Calls on another stream must come after the zeroing."""
    n = decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_context_len,
                               num_splits)
    if stream is None:
        return torch.zeros(max(n, 16), dtype=torch.uint8, device=device or "cuda")
    s = stream if isinstance(stream, torch.cuda.Stream) else torch.cuda.ExternalStream(int(stream))
    with torch.cuda.stream(s):
        return torch.zeros(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def paged_decode_attn(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_tables: torch.Tensor, context_lens: torch.Tensor,
                      max_context_len: int, scale: float, num_splits: int = 0,
                      workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """One query token per sequence over its paged KV (GQA). q: [B, Hq, D] bf16;
    caches [NB, bs, Hkv, D] bf16; block_tables [B, W] int32; context_lens [B] int32."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.bfloat16)
    _need(block_tables, "block_tables", torch.int32)
    _need(context_lens, "context_lens", torch.int32)
    if not (q.is_contiguous() and k_cache.is_contiguous() and v_cache.is_contiguous()
            and block_tables.is_contiguous() and context_lens.is_contiguous()):
        raise ValueError("q, caches, block_tables and context_lens must be contiguous")
    B, hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = decode_workspace(B, hq, hkv, d, max_context_len, num_splits, q.device,
                                     stream)
    _check("pkv_paged_decode_attn", _LIB.pkv_paged_decode_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), B, int(max_context_len), hq, hkv, d, bs, nb, float(scale),
        int(num_splits), _ptr(workspace), workspace.numel(), _ptr(out), _stream(stream)))
    return out


def paged_decode_step(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                      slot_mapping: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_tables: torch.Tensor, context_lens: torch.Tensor,
                      max_context_len: int, scale: float, num_splits: int = 0,
                      workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """Store each sequence's new token (k_new, v_new: [B, Hkv, D], rows may be strided views;
    slot_mapping [B] int64) and attend, in one call: the same result as kv_store followed by
    paged_decode_attn."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (k_new, "k_new"),
                 (v_new, "v_new")):
        _need(t, n, torch.bfloat16)
    _need(block_tables, "block_tables", torch.int32)
    _need(context_lens, "context_lens", torch.int32)
    _need(slot_mapping, "slot_mapping", torch.int64)
    if not (q.is_contiguous() and k_cache.is_contiguous() and v_cache.is_contiguous()
            and block_tables.is_contiguous() and context_lens.is_contiguous()
            and slot_mapping.is_contiguous()):
        raise ValueError("q, caches, block_tables, context_lens, slot_mapping must be contiguous")
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        if t.stride(-1) != 1 or t.stride(-2) != t.shape[-1]:
            raise ValueError(f"{n}: each token's heads must be dense")
    B, hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = decode_workspace(B, hq, hkv, d, max_context_len, num_splits, q.device,
                                     stream)
    _check("pkv_paged_decode_step", _LIB.pkv_paged_decode_step(
        _ptr(q), _ptr(k_new), k_new.stride(0), _ptr(v_new), v_new.stride(0), _ptr(slot_mapping),
        _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), B, int(max_context_len), hq, hkv, d, bs, nb, float(scale),
        int(num_splits), _ptr(workspace), workspace.numel(), _ptr(out), _stream(stream)))
    return out


def paged_decode_attn_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                              block_tables: torch.Tensor, context_lens: torch.Tensor,
                              max_context_len: int, scale: float, num_splits: int = 0,
                              out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """paged_decode_attn without a workspace argument, for callers that cannot allocate
    device memory: the split results go to a fixed array inside the library (see pkv.h).
    Calls on one device must not overlap on the GPU."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.bfloat16)
    _need(block_tables, "block_tables", torch.int32)
    _need(context_lens, "context_lens", torch.int32)
    if not (q.is_contiguous() and k_cache.is_contiguous() and v_cache.is_contiguous()
            and block_tables.is_contiguous() and context_lens.is_contiguous()):
        raise ValueError("q, caches, block_tables and context_lens must be contiguous")
    B, hq, d = q.shape
    nb, bs, hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    _check("pkv_paged_decode_attn_noalloc", _LIB.pkv_paged_decode_attn_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), B, int(max_context_len), hq, hkv, d, bs, nb, float(scale),
        int(num_splits), _ptr(out), _stream(stream)))
    return out


def varlen_prefill_attn(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                        cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor,
                        max_seqlen_q: int, max_seqlen_k: int, scale: float, causal: bool = True,
                        block_table: torch.Tensor | None = None,
                        out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """Causal attention over cu_seqlens-packed sequences. q: [Tq, Hq, D]; k, v: packed
    [Tk, Hkv, D], or the pools [NB, bs, Hkv, D] when block_table [N, W] int32 is given.
    workspace: pkv_prefill_workspace_bytes bytes (allocated per call when omitted)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32)
    tq, hq, d = q.shape
    if q.stride(2) != 1 or q.stride(1) != d:
        raise ValueError("q must have dense rows")
    if block_table is not None:
        _need(block_table, "block_table", torch.int32)
        nb, bs, hkv, _ = k.shape
        if not (k.is_contiguous() and v.is_contiguous() and block_table.is_contiguous()):
            raise ValueError("pools and block_table must be contiguous")
        kv_stride, total_k, W = hkv * d, 0, block_table.shape[1]
    else:
        total_k, hkv, _ = k.shape
        if k.stride() != v.stride() or k.stride(2) != 1 or k.stride(1) != d:
            raise ValueError("k and v must share a layout with dense rows")
        kv_stride, nb, bs, W = k.stride(0), 0, 0, 0
    if out is None:
        out = torch.empty((tq, hq, d), dtype=q.dtype, device=q.device)
    else:
        _need(out, "out", torch.bfloat16)
        if tuple(out.shape) != (tq, hq, d) or not out.is_contiguous():
            raise ValueError("out must be a contiguous [Tq, Hq, D] tensor")
    n = cu_seqlens_q.shape[0] - 1
    if workspace is None:
        workspace = torch.empty(max(16, int(_LIB.pkv_prefill_workspace_bytes(n, int(max_seqlen_q),
                                                                          hq, d))),
                                dtype=torch.uint8, device=q.device)
    _check("pkv_varlen_prefill_attn", _LIB.pkv_varlen_prefill_attn(
        _ptr(q), q.stride(0), tq, _ptr(k), _ptr(v), kv_stride, total_k,
        _ptr(cu_seqlens_q.contiguous()), _ptr(cu_seqlens_k.contiguous()), n, int(max_seqlen_q),
        int(max_seqlen_k), _ptr(block_table), W, bs, nb, hq, hkv, d, float(scale),
        int(bool(causal)), _ptr(workspace), workspace.numel(), _ptr(out), _stream(stream)))
    return out


def qk_norm_rope_store(qkv, positions, q_norm_weight, k_norm_weight, eps, cos_sin_cache,
                       slot_mapping, k_cache, v_cache, num_q_heads: int, num_kv_heads: int,
                       q_out=None, stream=None):
    """QK RMSNorm + RoPE of the new tokens, K/V stored into the pool, q returned.

    qkv: [T, (Hq + 2 Hkv) * D] bf16 (rows may be a strided view); positions, slot_mapping:
    [T] int64; weights [D] bf16; cos_sin_cache [max_position, D] float32; pools
    [NB, bs, Hkv, D] bf16. Returns q [T, Hq, D] bf16."""
    T = qkv.shape[0]
    D = q_norm_weight.shape[0]
    assert qkv.dtype == torch.bfloat16 and qkv.is_cuda and qkv.stride(-1) == 1
    for t in (q_norm_weight, k_norm_weight, k_cache, v_cache):
        assert t.dtype == torch.bfloat16 and t.is_cuda and t.is_contiguous()
    assert cos_sin_cache.dtype == torch.float32 and cos_sin_cache.is_contiguous()
    assert positions.dtype == torch.int64 and slot_mapping.dtype == torch.int64
    positions, slot_mapping = positions.contiguous(), slot_mapping.contiguous()
    if q_out is None:
        q_out = torch.empty((T, num_q_heads, D), dtype=torch.bfloat16, device=qkv.device)
    num_slots = k_cache.numel() // (num_kv_heads * D)
    _check("pkv_qk_norm_rope_store", _LIB.pkv_qk_norm_rope_store(
        qkv.data_ptr(), qkv.stride(0) if T else qkv.shape[-1], T, positions.data_ptr(),
        q_norm_weight.data_ptr(), k_norm_weight.data_ptr(), float(eps),
        cos_sin_cache.data_ptr(), cos_sin_cache.shape[0], slot_mapping.data_ptr(),
        q_out.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), num_slots, num_q_heads,
        num_kv_heads, D, _stream(stream)))
    return q_out


# ----------------------------------------------------------------------------- block manager
def xxh64(data: bytes, seed: int = 0) -> int:
    """XXH64 of a byte string, computed by the library (the block manager's hash)."""
    buf = ctypes.create_string_buffer(bytes(data), max(1, len(data)))
    return int(_LIB.pkv_xxh64(buf, len(data), seed))


class BlockManager:
    """Host-side block manager of libpkv (pkv_bm_* in include/pkv.h): blocks with reference
    counts and prefix-cache hashes. Sequences are lists of int token ids; block tables are
    lists of block ids. Every call goes to the C++ implementation."""

    def __init__(self, num_blocks: int, block_size: int):
        h = _LIB.pkv_bm_create(int(num_blocks), int(block_size))
        if not h:
            raise PkvError("pkv_bm_create", ERR_INVALID_ARG)
        self._h = ctypes.c_void_p(h)
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            _LIB.pkv_bm_destroy(h)
            self._h = None

    @staticmethod
    def _ints(xs):
        xs = list(xs)
        return (ctypes.c_int32 * max(1, len(xs)))(*xs), len(xs)

    @property
    def num_free(self) -> int:
        return int(_LIB.pkv_bm_num_free(self._h))

    def ref_count(self, block: int) -> int:
        return int(_LIB.pkv_bm_ref_count(self._h, int(block)))

    def block_hash(self, block: int):
        """The block's hash, or None while it is not full and registered."""
        h, ok = ctypes.c_uint64(), ctypes.c_int32()
        _check("pkv_bm_block_hash", _LIB.pkv_bm_block_hash(self._h, int(block),
                                                             ctypes.byref(h), ctypes.byref(ok)))
        return int(h.value) if ok.value else None

    def allocate(self, token_ids):
        """Block table and number of cached leading tokens for a new sequence."""
        toks, n = self._ints(token_ids)
        cap = max(1, -(-n // self.block_size))
        table = (ctypes.c_int32 * cap)()
        nb, cached = ctypes.c_int32(), ctypes.c_int32()
        _check("pkv_bm_allocate", _LIB.pkv_bm_allocate(self._h, toks, n, table, cap,
                                                       ctypes.byref(nb), ctypes.byref(cached)))
        return list(table[:nb.value]), int(cached.value)

    def deallocate(self, table) -> None:
        t, n = self._ints(table)
        _check("pkv_bm_deallocate", _LIB.pkv_bm_deallocate(self._h, t, n))

    def can_append(self, seq_len: int) -> bool:
        return bool(_LIB.pkv_bm_can_append(self._h, int(seq_len)))

    def may_append(self, token_ids, table):
        """After appending a token (token_ids = the whole sequence): the updated table."""
        toks, n = self._ints(token_ids)
        cap = len(table) + 1
        t = (ctypes.c_int32 * cap)(*table)
        nb = ctypes.c_int32(len(table))
        _check("pkv_bm_may_append", _LIB.pkv_bm_may_append(self._h, toks, n, t, cap,
                                                           ctypes.byref(nb)))
        return list(t[:nb.value])
