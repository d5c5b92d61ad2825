"""Golden fixtures (tests/golden/, written by make_golden.py from the oracle): the oracle must
keep reproducing them (a change to its arithmetic shows up here), and the GPU kernels must
match them within the attention tolerance."""
import os

import numpy as np
import pytest

import oracle
import workloads as w
from tests_golden_util import load_fixture

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _tiny_decode():
    lay, val = w.tiny_decode()
    kc, vc = val.k_cache.copy(), val.v_cache.copy()
    oracle.kv_store(val.k_new, val.v_new, lay.slot_mapping, kc, vc)
    return lay, val, oracle.paged_decode(val.q, kc, vc, lay.block_tables, lay.context_lens,
                                         lay.scale)


def test_oracle_reproduces_tiny_decode_fixture():
    rows = load_fixture(os.path.join(HERE, "tiny_decode.txt"))
    _, _, out = _tiny_decode()
    for (b, hq), vals in rows.items():
        got = [out[b, hq].sum()] + [out[b, hq, d] for d in (0, 1, 64, 127)]
        np.testing.assert_allclose(got, vals, rtol=1e-13, atol=1e-13)


def test_oracle_reproduces_small_prefill_fixture():
    rows = load_fixture(os.path.join(HERE, "small_prefill.txt"))
    g = w.rng(3)
    lay = w.prefill_layout([100, 257, 31], 8, g)
    val = w.prefill_values(lay, g)
    cu = lay.cu_seqlens_q
    out = oracle.varlen_prefill(val.q, val.k, val.v, cu, cu, lay.scale)
    for (t, hq), vals in rows.items():
        got = [out[t, hq].sum(), out[t, hq, 0], out[t, hq, 127]]
        np.testing.assert_allclose(got, vals, rtol=1e-13, atol=1e-13)


@pytest.mark.gpu
def test_gpu_decode_matches_tiny_decode_fixture():
    from gpu_util import dev, host_f64
    from libbuild import build_and_import
    pkv = build_and_import()
    rows = load_fixture(os.path.join(HERE, "tiny_decode.txt"))
    lay, val = w.tiny_decode()
    kc, vc = dev(val.k_cache), dev(val.v_cache)
    pkv.kv_store(dev(val.k_new), dev(val.v_new), dev(lay.slot_mapping), kc, vc)
    out = host_f64(pkv.paged_decode_attn(dev(val.q), kc, vc, dev(lay.block_tables),
                                         dev(lay.context_lens), lay.max_context_len, lay.scale))
    for (b, hq), vals in rows.items():
        got = np.array([out[b, hq, d] for d in (0, 1, 64, 127)])
        ref = np.array(vals[1:])
        assert (np.abs(got - ref) <= 1e-2 + 1e-2 * np.abs(ref)).all(), (b, hq)
