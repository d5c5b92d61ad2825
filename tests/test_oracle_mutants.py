"""Plant plausible mistakes in copies of the oracle and check that its pins catch each one.

Every mutant is one textual change to a copy of ``oracle/pkv_oracle.c``, compiled with gcc
into a temporary library; the shipped oracle source is never touched. A mutant survives if
every pin in ``oracle_pins`` still passes, which would mean the pins cannot tell that mistake
from the right answer. None of the mutants reads or writes out of bounds. The block manager
oracle (``oracle/block_manager.py``, plain Python) gets the same treatment against the pins in
``block_manager_pins``, each mutant loaded from a temporary copy.
"""
import os
import shutil

import pytest

import oracle
import oracle_pins
from oracle import build as obuild

# (name, original text, replacement, which occurrence (0-based) or None for all)
MUTANTS = [
    ("dropped_scale", "score[j] = scale * dot;", "score[j] = dot;", None),
    ("exp_sign_flipped", "score[j] = exp(score[j] - m);", "score[j] = exp(m - score[j]);", None),
    ("max_not_subtracted", "score[j] = exp(score[j] - m);", "score[j] = exp(score[j]);", None),
    ("max_starts_at_zero", "double m = score[0];", "double m = 0.0;", None),
    ("denominator_dropped", "out[d] /= denom;", "out[d] /= 1.0;", None),
    ("keys_read_from_v", "const uint16_t *kj = k_base + key_rows[j];",
     "const uint16_t *kj = v_base + key_rows[j];", None),
    ("values_read_from_k", "const uint16_t *vj = v_base + key_rows[j];",
     "const uint16_t *vj = k_base + key_rows[j];", None),
    ("decode_gqa_interleaved", "const int32_t h = hq / group;",
     "const int32_t h = hq % num_kv_heads;", 0),
    ("prefill_gqa_interleaved", "const int32_t h = hq / group;",
     "const int32_t h = hq % num_kv_heads;", 1),
    ("decode_offset_from_block_index", "const int64_t slot = blk * block_size + i % block_size;",
     "const int64_t slot = blk * block_size + (i / block_size) % block_size;", None),
    ("decode_drops_newest_token", "rows, L, head_dim, scale, score, o);",
     "rows, L > 1 ? L - 1 : L, head_dim, scale, score, o);", None),
    ("prefill_paged_offset_wrong", "key_row = blk * block_size + j % block_size;",
     "key_row = blk * block_size + (j + 1) % block_size;", None),
    ("causal_top_left", "int64_t visible = causal ? i + (Lk - Lq) + 1 : Lk;",
     "int64_t visible = causal ? i + 1 : Lk;", None),
    ("causal_excludes_diagonal", "int64_t visible = causal ? i + (Lk - Lq) + 1 : Lk;",
     "int64_t visible = causal ? i + (Lk - Lq) : Lk;", None),
    ("causal_ignored", "int64_t visible = causal ? i + (Lk - Lq) + 1 : Lk;",
     "int64_t visible = Lk;", None),
    ("store_v_into_k", "k_cache[slot * row + e] = k[t * k_tok_stride + e];",
     "k_cache[slot * row + e] = v[t * v_tok_stride + e];", None),
    ("store_ignores_token_stride", "k_cache[slot * row + e] = k[t * k_tok_stride + e];",
     "k_cache[slot * row + e] = k[t * row + e];", None),
    ("store_skips_duplicate_check", "if (seen[slot]) { free(seen); return ORACLE_DUP_SLOT; }",
     "", None),
    ("rms_sum_not_mean", "1.0 / sqrt(ss / head_dim + eps)", "1.0 / sqrt(ss + eps)", None),
    ("rms_eps_dropped", "1.0 / sqrt(ss / head_dim + eps)", "1.0 / sqrt(ss / head_dim)", None),
    ("norm_weight_dropped", "n[d] = bf16_value(x[d]) * r * bf16_value(w[d]);",
     "n[d] = bf16_value(x[d]) * r;", None),
    ("rope_sin_sign_flipped", "y[i + half] = n[i + half] * c + n[i] * sn;",
     "y[i + half] = n[i + half] * c - n[i] * sn;", None),
    ("rope_cos_sin_swapped", "const double c = cs[i], sn = cs[half + i];",
     "const double c = cs[half + i], sn = cs[i];", None),
    ("rope_pairs_adjacent", "y[i] = n[i] * c - n[i + half] * sn;",
     "y[i] = n[i] * c - n[i ^ 1] * sn;", None),
]


def _mutate(src: str, old: str, new: str, occurrence):
    n = src.count(old)
    assert n >= 1, f"mutation anchor not found: {old!r}"
    if occurrence is None:
        return src.replace(old, new)
    assert occurrence < n
    pos = -1
    for _ in range(occurrence + 1):
        pos = src.index(old, pos + 1)
    return src[:pos] + new + src[pos + len(old):]


@pytest.mark.parametrize("name,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, occ):
    src = open(obuild.SRC).read()
    path = tmp_path / f"{name}.c"
    path.write_text(_mutate(src, old, new, occ))
    lib_path = obuild.build(str(path), str(tmp_path / f"lib{name}.so"), force=True)
    L = oracle.load(lib_path)
    failures = []
    for pin in oracle_pins.ALL_PINS:
        try:
            oracle_pins.run_pin(pin, L)
        except (AssertionError, oracle.OracleError) as e:
            failures.append(pin.__name__)
    assert failures, f"mutant {name} survives every pin"


def test_unmutated_copy_passes(tmp_path):
    path = tmp_path / "copy.c"
    shutil.copy(obuild.SRC, path)
    L = oracle.load(obuild.build(str(path), str(tmp_path / "libcopy.so"), force=True))
    for pin in oracle_pins.ALL_PINS:
        oracle_pins.run_pin(pin, L)


# ------------------------------------------------------------- the block manager oracle
# Plausible mistakes in oracle/block_manager.py, each of which must fail at least one of its
# pins (tests/block_manager_pins.py).
BM_MUTANTS = [
    ("xxh64_prime_typo", "0xC2B2AE3D27D4EB4F", "0xC2B2AE3D27D4EB4E", None),
    ("xxh64_tail4_wrong_prime", 'h ^= (int.from_bytes(data[i:i + 4], "little") * P1) & M64',
     'h ^= (int.from_bytes(data[i:i + 4], "little") * P2) & M64', None),
    ("xxh64_no_avalanche_shift", "h ^= h >> 33", "h ^= h >> 0", None),
    ("xxh64_length_not_added", "h = (h + n) & M64", "h = h & M64", None),
    ("hash_not_chained", 'data = b"" if prefix is None else prefix.to_bytes(8, "little")',
     'data = b""', None),
    ("hash_tokens_8_bytes", '(t & 0xFFFFFFFF).to_bytes(4, "little")',
     '(t & 0xFFFFFFFF).to_bytes(8, "little")', None),
    ("free_list_lifo", "b = self.free.pop(0)", "b = self.free.pop()", None),
    ("hit_without_token_check", "if b is not None and self.tokens[b] == toks:",
     "if b is not None:", None),
    ("dealloc_first_block_first", "for b in reversed(table):", "for b in table:", None),
    ("no_upfront_block_check", "if len(self.free) < len(blocks):", "if False:", None),
    ("append_hashes_wrong_block", "if n % bs == 0:", "if n % bs == 1:", None),
    ("cached_blocks_not_counted", "cached += bs", "cached += 0", None),
]


def _load_module(path, name):
    import importlib.util
    spec = importlib.util.spec_from_file_location(name, path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name,old,new,occ", BM_MUTANTS, ids=[m[0] for m in BM_MUTANTS])
def test_block_manager_mutant_is_caught(tmp_path, name, old, new, occ):
    import block_manager_pins
    src = open(os.path.join(os.path.dirname(oracle.__file__), "block_manager.py")).read()
    path = tmp_path / f"bm_{name}.py"
    path.write_text(_mutate(src, old, new, occ))
    mod = _load_module(str(path), f"bm_mutant_{name}")
    failures = []
    for pin in block_manager_pins.ALL_PINS:
        try:
            pin(mod)
        except Exception:  # an assertion, or the mutant crashing on the pin's inputs
            failures.append(pin.__name__)
    assert failures, f"block manager mutant {name} survives every pin"


def test_block_manager_unmutated_copy_passes(tmp_path):
    import block_manager_pins
    src = os.path.join(os.path.dirname(oracle.__file__), "block_manager.py")
    path = tmp_path / "bm_copy.py"
    shutil.copy(src, path)
    mod = _load_module(str(path), "bm_copy")
    for pin in block_manager_pins.ALL_PINS:
        pin(mod)
