"""The C-ABI library loads and exports every symbol include/pkv.h declares; host-side
argument checks return their status codes without touching a GPU (no compute calls)."""
import ctypes
import os
import re

import pytest

from libbuild import ROOT, build_and_import

pkv = build_and_import()
L = pkv.lib()
FAKE = ctypes.c_void_p(0x1000)   # never dereferenced: every call below fails or returns early


def header_functions():
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = header_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(L, n), f"{n} declared in pkv.h but not exported"
    assert sorted(pkv.SIGNATURES) == names, "binding signatures out of step with pkv.h"


def test_status_strings():
    for code in range(5):
        assert L.pkv_status_string(code)
    assert L.pkv_status_string(99) == b"unknown status"
    assert L.pkv_abi_version() == 2


def test_store_argument_checks():
    s = L.pkv_kv_store
    assert s(FAKE, 1024, FAKE, 1024, FAKE, 0, FAKE, FAKE, 10, 8, 128, None) == pkv.OK
    assert s(FAKE, 1024, FAKE, 1024, FAKE, -1, FAKE, FAKE, 10, 8, 128, None) == pkv.ERR_INVALID_ARG
    assert s(FAKE, 512, FAKE, 1024, FAKE, 4, FAKE, FAKE, 10, 8, 128, None) == pkv.ERR_INVALID_ARG
    assert s(None, 1024, FAKE, 1024, FAKE, 4, FAKE, FAKE, 10, 8, 128, None) == pkv.ERR_INVALID_ARG
    assert s(FAKE, 1024, FAKE, 1024, FAKE, 4, FAKE, FAKE, -1, 8, 128, None) == pkv.ERR_INVALID_ARG
    assert s(FAKE, 1024, FAKE, 1024, FAKE, 4, FAKE, FAKE, 10, 0, 128, None) == pkv.ERR_INVALID_ARG


def _decode(**kw):
    a = dict(q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, W=4, cl=FAKE, B=2, maxc=100, hq=16, hkv=8, d=128,
             bs=256, nb=10, scale=0.088, ns=0, ws=FAKE, wsb=1 << 20, out=FAKE)
    a.update(kw)
    return L.pkv_paged_decode_attn(a["q"], a["kc"], a["vc"], a["bt"], a["W"], a["cl"], a["B"],
                                   a["maxc"], a["hq"], a["hkv"], a["d"], a["bs"], a["nb"],
                                   a["scale"], a["ns"], a["ws"], a["wsb"], a["out"], None)


def test_decode_argument_checks():
    assert _decode(B=0) == pkv.OK
    assert _decode(B=-1) == pkv.ERR_INVALID_ARG
    assert _decode(hq=12, hkv=8) == pkv.ERR_INVALID_ARG
    assert _decode(q=None) == pkv.ERR_INVALID_ARG
    assert _decode(scale=float("nan")) == pkv.ERR_INVALID_ARG
    assert _decode(ns=-2) == pkv.ERR_INVALID_ARG
    assert _decode(W=0) == pkv.ERR_INVALID_ARG
    assert _decode(d=64) == pkv.ERR_UNSUPPORTED
    assert _decode(bs=16) == pkv.ERR_UNSUPPORTED
    assert _decode(nb=1 << 24) == pkv.ERR_UNSUPPORTED          # rows beyond int32
    assert _decode(q=ctypes.c_void_p(0x1008)) == pkv.ERR_UNSUPPORTED  # not 16-byte aligned


def _prefill(**kw):
    a = dict(q=FAKE, qs=2048, tq=100, k=FAKE, v=FAKE, kvs=1024, tk=100, cq=FAKE, ck=FAKE, N=2,
             mq=64, mk=64, bt=None, W=0, bs=0, nb=0, hq=16, hkv=8, d=128, scale=0.088, causal=1,
             ws=FAKE, wsb=1 << 20, out=FAKE)
    a.update(kw)
    return L.pkv_varlen_prefill_attn(a["q"], a["qs"], a["tq"], a["k"], a["v"], a["kvs"], a["tk"],
                                     a["cq"], a["ck"], a["N"], a["mq"], a["mk"], a["bt"], a["W"],
                                     a["bs"], a["nb"], a["hq"], a["hkv"], a["d"], a["scale"],
                                     a["causal"], a["ws"], a["wsb"], a["out"], None)


def test_prefill_argument_checks():
    assert _prefill(N=0) == pkv.OK
    assert _prefill(tq=0) == pkv.OK
    assert _prefill(N=-1) == pkv.ERR_INVALID_ARG
    assert _prefill(qs=1000) == pkv.ERR_INVALID_ARG               # shorter than a q row
    assert _prefill(kvs=512) == pkv.ERR_INVALID_ARG
    assert _prefill(cq=None) == pkv.ERR_INVALID_ARG
    assert _prefill(bt=FAKE, W=0, bs=256, nb=4) == pkv.ERR_INVALID_ARG
    assert _prefill(d=64, qs=1024, kvs=512) == pkv.ERR_UNSUPPORTED
    assert _prefill(bt=FAKE, W=4, bs=128, nb=4) == pkv.ERR_UNSUPPORTED
    assert _prefill(bt=FAKE, W=4, bs=256, nb=4, kvs=2048) == pkv.ERR_UNSUPPORTED
    assert _prefill(qs=2052) == pkv.ERR_UNSUPPORTED                # stride not 16-byte multiple
    assert _prefill(ws=None) == pkv.ERR_WORKSPACE
    assert _prefill(wsb=8) == pkv.ERR_WORKSPACE
    need = L.pkv_prefill_workspace_bytes(2, 64, 16, 128)
    assert _prefill(wsb=need - 16) == pkv.ERR_WORKSPACE            # the work list does not fit


def _step(**kw):
    a = dict(q=FAKE, kn=FAKE, kns=1024, vn=FAKE, vns=1024, slots=FAKE, kc=FAKE, vc=FAKE, bt=FAKE,
             W=4, cl=FAKE, B=2, maxc=100, hq=16, hkv=8, d=128, bs=256, nb=10, scale=0.088, ns=0,
             ws=FAKE, wsb=1 << 20, out=FAKE)
    a.update(kw)
    return L.pkv_paged_decode_step(a["q"], a["kn"], a["kns"], a["vn"], a["vns"], a["slots"],
                                   a["kc"], a["vc"], a["bt"], a["W"], a["cl"], a["B"], a["maxc"],
                                   a["hq"], a["hkv"], a["d"], a["bs"], a["nb"], a["scale"],
                                   a["ns"], a["ws"], a["wsb"], a["out"], None)


def test_decode_step_argument_checks():
    assert _step(B=0) == pkv.OK
    assert _step(B=-1) == pkv.ERR_INVALID_ARG
    assert _step(kns=512) == pkv.ERR_INVALID_ARG                   # new K rows shorter than Hkv*D
    assert _step(slots=None) == pkv.ERR_INVALID_ARG
    assert _step(hq=12, hkv=8) == pkv.ERR_INVALID_ARG
    assert _step(scale=float("inf")) == pkv.ERR_INVALID_ARG
    assert _step(d=64, kns=512, vns=512) == pkv.ERR_UNSUPPORTED
    assert _step(bs=128) == pkv.ERR_UNSUPPORTED
    assert _step(kns=1028) == pkv.ERR_UNSUPPORTED                  # stride not a 16-byte multiple
    assert _step(vn=ctypes.c_void_p(0x1008)) == pkv.ERR_UNSUPPORTED  # not 16-byte aligned


def _rope(**kw):
    a = dict(qkv=FAKE, ts=4096, T=4, pos=FAKE, qw=FAKE, kw=FAKE, eps=1e-6, cs=FAKE, maxp=1024,
             slots=FAKE, q=FAKE, kc=FAKE, vc=FAKE, nslots=512, hq=16, hkv=8, d=128)
    a.update(kw)
    return L.pkv_qk_norm_rope_store(a["qkv"], a["ts"], a["T"], a["pos"], a["qw"], a["kw"],
                                    a["eps"], a["cs"], a["maxp"], a["slots"], a["q"], a["kc"],
                                    a["vc"], a["nslots"], a["hq"], a["hkv"], a["d"], None)


def test_qk_norm_rope_store_argument_checks():
    assert _rope(T=0) == pkv.OK
    assert _rope(T=-1) == pkv.ERR_INVALID_ARG
    assert _rope(ts=4000) == pkv.ERR_INVALID_ARG                   # shorter than a projection row
    assert _rope(eps=float("nan")) == pkv.ERR_INVALID_ARG
    assert _rope(eps=-1.0) == pkv.ERR_INVALID_ARG
    assert _rope(maxp=0) == pkv.ERR_INVALID_ARG
    assert _rope(pos=None) == pkv.ERR_INVALID_ARG
    assert _rope(d=64, ts=2048) == pkv.ERR_UNSUPPORTED
    assert _rope(ts=4100) == pkv.ERR_UNSUPPORTED                   # stride not a 16-byte multiple
    assert _rope(q=ctypes.c_void_p(0x1008)) == pkv.ERR_UNSUPPORTED  # not 16-byte aligned


def test_workspace_query_without_device_is_zero_or_sized():
    n = L.pkv_decode_workspace_bytes(4, 16, 8, 128, 300, 0)
    assert n == 0 or n >= 16   # 0 without a device to plan for
    assert L.pkv_decode_workspace_bytes(4, 16, 8, 64, 300, 0) == 0
    # a header and sort arrays, then one 8-byte unit per (sequence, 128-query block) at most
    for n, L_q in ((4, 100), (256, 1024), (1, 131072), (0, 0)):
        b = L.pkv_prefill_workspace_bytes(n, L_q, 16, 128)
        assert b % 16 == 0 and b >= 16 + 8 * n * (-(-L_q // 128)), (n, L_q, b)
        assert b <= 16 + 8 * n * (-(-L_q // 128)) + 32 * (n + 1) + 16 * (-(-L_q // 128) + 1) + 96
    assert L.pkv_prefill_workspace_bytes(-1, 100, 16, 128) == 0
    assert L.pkv_prefill_workspace_bytes(100000, 2 ** 30, 16, 128) == 0   # list too long


def test_product_path_has_no_oracle_import():
    """The package must not reach the CPU oracle: no import of it anywhere in its sources."""
    pkg = os.path.join(ROOT, "paged_kv_cache_208_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cc", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower().replace("the oracle", ""), f
