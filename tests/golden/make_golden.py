"""Write the golden fixtures of this directory from the CPU oracle (and nothing else).

    python tests/golden/make_golden.py

tiny_decode.txt   -- the tiny decode step (contexts {1, 17, 255, 300}, pool of 8 blocks in a
                     seeded permutation; the decode configuration of the nano-vLLM pages:
                     «nano-vLLM 最小化vLLM重新实现» 架构 5, decode over the paged cache with
                     block tables and cache lengths): the oracle's output for every
                     (sequence, query head), as the sum over head_dim and 4 sampled values.
small_prefill.txt -- varlen causal prefill over prompts {100, 257, 31} (架构 5, prefill with
                     flash_attn_varlen_func): per (token, head) sums and 2 sampled values.
Values are printed with 17 significant digits (round-trips float64).
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import workloads as w  # noqa: E402

DIMS = (0, 1, 64, 127)


def tiny_decode_lines():
    lay, val = w.tiny_decode()
    kc, vc = val.k_cache.copy(), val.v_cache.copy()
    oracle.kv_store(val.k_new, val.v_new, lay.slot_mapping, kc, vc)
    out = oracle.paged_decode(val.q, kc, vc, lay.block_tables, lay.context_lens, lay.scale)
    lines = ["# tiny decode step, seed 1: b hq sum(out[b,hq,:]) out[b,hq,0] out[b,hq,1] "
             "out[b,hq,64] out[b,hq,127]"]
    for b in range(out.shape[0]):
        for hq in range(out.shape[1]):
            vals = [out[b, hq].sum()] + [out[b, hq, d] for d in DIMS]
            lines.append(f"{b} {hq} " + " ".join(f"{x:.17g}" for x in vals))
    return lines


def small_prefill_lines():
    g = w.rng(3)
    lay = w.prefill_layout([100, 257, 31], 8, g)
    val = w.prefill_values(lay, g)
    cu = lay.cu_seqlens_q
    out = oracle.varlen_prefill(val.q, val.k, val.v, cu, cu, lay.scale)
    lines = ["# varlen causal prefill {100, 257, 31}, seed 3: t hq sum(out[t,hq,:]) "
             "out[t,hq,0] out[t,hq,127]"]
    for t in range(0, out.shape[0], 7):
        for hq in (0, 5, 15):
            vals = [out[t, hq].sum(), out[t, hq, 0], out[t, hq, 127]]
            lines.append(f"{t} {hq} " + " ".join(f"{x:.17g}" for x in vals))
    return lines


def main():
    for name, fn in (("tiny_decode.txt", tiny_decode_lines), ("small_prefill.txt",
                                                               small_prefill_lines)):
        with open(os.path.join(HERE, name), "w") as f:
            f.write("\n".join(fn()) + "\n")


if __name__ == "__main__":
    main()
