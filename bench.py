"""Benchmark of the paged KV cache hot path on GB300.

One step = one decode step of a Qwen3-0.6B-shaped model over its 28 layers: for each layer,
kv_store of the 256 sequences' new K/V into that layer's block pool, then paged decode
attention of the 256 queries over contexts drawn uniform in [100, 2048] (blocks drawn at
random from a pool sized to 90% of free HBM). Inputs are synthetic and already in HBM when
the timed region starts; every layer reads 1.13 GB of KV, far more than the 129 MB L2.

The JSON line reports the step's algorithmic HBM bytes per second (value), KV-tokens/s, the
decode kernel's roofline fraction, the same metric end to end through the public API with
host buffers (e2e), the varlen-prefill store's GB/s and the prefill TFLOP/s measured in the
same run, and the CPU oracle timed on the host cores as a baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With N > 1 (torchrun, one process per GPU) every rank runs its own full batch (weak scaling;
no data-path collective) and rank 0 prints the line; value = bytes of all ranks / max time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as w  # noqa: E402

METRIC = ("paged decode attn HBM GB/s (% of peak) & KV-tokens/s; kv_store GB/s; "
          "prefill TFLOP/s")
LAYERS = w.NUM_LAYERS
B, HQ, HKV, D, BS = 256, w.NUM_Q_HEADS, w.NUM_KV_HEADS, w.HEAD_DIM, w.BLOCK_SIZE
ROW_BYTES = HKV * D * 2                     # one token's K (or V) row in one layer
BLOCK_BYTES_ALL_LAYERS = 2 * LAYERS * BS * ROW_BYTES
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# The committed ncu summary of decode_split_kernel on the Qwen3 decode batch. It records the
# DRAM bytes of one launch and a hash of the kernel's sources at the time of the capture; the
# bench reports that traffic only while the sources still hash the same.
DECODE_PROFILE = os.path.join(ROOT, "profiles", "decode_split_qwen3_decode_batch.md")
DECODE_SOURCES = ("paged_kv_cache_208_gb300/csrc/decode.cu",
                  "paged_kv_cache_208_gb300/csrc/device_common.cuh")
MIN_TIMED_SECONDS = 2.0   # the headline's K-step blocks are repeated until they cover this
WORKLOAD = ("qwen3-0.6b decode step: 28 layers x (kv_store of 256 new tokens + paged decode "
            "attention), B=256, ctx U[100,2048] (seed 2), block_size 256, 16 q / 8 kv heads, "
            "head_dim 128, bf16 N(0,1), pool [2,28,NB,256,8,128] at 90% of free HBM")


# ----------------------------------------------------------------------------- helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        hbm = d.get("hbm_gbs") or d.get("hbm_GBps") or d.get("hbm")
        bf16 = d.get("bf16_tflops") or d.get("bf16")
        sus = d.get("bf16_tflops_sustained") or bf16
        if hbm:
            return float(hbm), float(bf16 or FALLBACK_BF16_TFLOPS), float(sus or 0), "measured"
    except (OSError, ValueError, TypeError):
        pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def sources_sha256(paths) -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def decode_traffic():
    """(DRAM bytes per launch, note) from the committed decode profile: the bytes are None
    when the profile is missing or the kernel's sources changed after the capture."""
    fields = {}
    try:
        with open(DECODE_PROFILE) as f:
            for line in f:
                if line.startswith("- ") and ": " in line:
                    k, v = line[2:].split(": ", 1)
                    fields[k.strip()] = v.strip().strip("`")
    except OSError:
        return None, "no committed profile"
    try:
        nbytes = int(fields["dram_bytes_per_launch"])
        sha = fields["sources_sha256"]
    except (KeyError, ValueError):
        return None, "profile has no machine-readable traffic line"
    if sha != sources_sha256(DECODE_SOURCES):
        return None, "kernel sources changed since the ncu capture"
    return nbytes, f"ncu capture in {os.path.relpath(DECODE_PROFILE, ROOT)} (sources {sha[:12]})"


def dist_env():
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    return rank, world, local


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Timing reduction only (no data-path collective): the slowest rank's time."""
    if world == 1:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def decode_bytes(ctx: np.ndarray, W: int) -> dict:
    """Algorithmic HBM bytes of one layer: the store and the decode call."""
    Bn = len(ctx)
    store = Bn * 2 * ROW_BYTES * 2 + Bn * 8                     # read k,v + write rows + slots
    decode = (int(ctx.sum()) * 2 * ROW_BYTES + 2 * Bn * HQ * D * 2 + 4 * Bn + 4 * Bn * W)
    return {"store": store, "decode": decode}


# --------------------------------------------------------------------------- decode step
class DecodeStep:
    def __init__(self, pkv, seed: int = 2, pool_fraction: float = 0.9, batch: int = B,
                 num_blocks: int | None = None, rank: int = 0, world: int = 1,
                 layers: int = LAYERS, num_splits: int = 0):
        self.pkv = pkv
        self.layers = layers
        self.num_splits = num_splits
        free, _ = torch.cuda.mem_get_info()
        ctx = w.qwen3_decode_lengths(seed, batch, rank=rank, world=world)
        need = w.blocks_needed(ctx)
        self.num_blocks = (int(pool_fraction * free // BLOCK_BYTES_ALL_LAYERS)
                           if num_blocks is None else num_blocks)
        if self.num_blocks < need:
            raise RuntimeError(f"pool of {self.num_blocks} blocks < {need} needed")
        self.lay = w.qwen3_decode_layout(self.num_blocks, seed, batch, rank, world)
        lay = self.lay
        self.B = lay.batch
        self.pool = torch.empty((2, layers, self.num_blocks, BS, HKV, D), dtype=torch.bfloat16,
                                device="cuda")
        ids = torch.from_numpy(np.unique(lay.block_tables[lay.block_tables >= 0])).long().cuda()
        for l in range(layers):      # only referenced blocks hold data (untimed)
            for kv in range(2):
                self.pool[kv, l][ids] = w.device_bf16_normal((len(ids), BS, HKV, D),
                                                             10_000 + 2 * l + kv)
        self.q = w.device_bf16_normal((layers, self.B, HQ, D), 20_001)
        self.kn = w.device_bf16_normal((layers, self.B, HKV, D), 20_002)
        self.vn = w.device_bf16_normal((layers, self.B, HKV, D), 20_003)
        self.out = torch.empty_like(self.q)
        self.slots = torch.from_numpy(lay.slot_mapping).cuda()
        self.tables = torch.from_numpy(lay.block_tables).cuda()
        self.ctx = torch.from_numpy(lay.context_lens).cuda()
        self.maxc = lay.max_context_len
        self.ws = pkv.decode_workspace(self.B, HQ, HKV, D, self.maxc, num_splits)
        self.splits_workspace = pkv.decode_workspace_bytes(self.B, HQ, HKV, D, self.maxc,
                                                           num_splits)
        self.bytes = decode_bytes(lay.context_lens, lay.block_tables.shape[1])
        self.step_bytes = layers * (self.bytes["store"] + self.bytes["decode"])
        self.kv_tokens = layers * int(lay.context_lens.sum())

    IO = ("q", "kn", "vn", "slots", "tables", "ctx")

    def run(self, events=None, io=None):
        """One step: per layer the store of the new tokens, then paged decode. `io` may give
        another set of the step's device inputs and output (q, kn, vn, slots, tables, ctx,
        out)."""
        pkv, s = self.pkv, self.pool
        io = io or {n: getattr(self, n) for n in self.IO + ("out",)}
        for l in range(self.layers):
            if events is not None:
                events.append(torch.cuda.Event(enable_timing=True))
                events[-1].record()
            # the layer's new tokens stored and attended in one call
            pkv.paged_decode_step(io["q"][l], io["kn"][l], io["vn"][l], io["slots"], s[0, l],
                                  s[1, l], io["tables"], io["ctx"], self.maxc, self.lay.scale,
                                  num_splits=self.num_splits, workspace=self.ws,
                                  out=io["out"][l])
            if events is not None:
                events.append(torch.cuda.Event(enable_timing=True))
                events[-1].record()

    def launches_per_step(self):
        # the split kernel (which also stores the new tokens), + the combine kernel when the
        # context is split (the workspace then holds partial outputs beyond its 16-byte counter)
        return self.layers * (1 + (1 if self.splits_workspace > 16 else 0))


def time_e2e(step: DecodeStep, steps: int):
    """The same step through the public API with host buffers, as a serving loop runs it:
    every step copies its inputs (q, k, v of 28 layers, slot_mapping, block_tables,
    context_lens) from pinned host memory and reads its 28 layers' outputs back, all inside the
    timed region. The copies run on a second stream into two alternating sets of device
    buffers, so step i+1's inputs arrive while step i computes and step i's output is read
    while step i+1 computes."""
    names = DecodeStep.IO
    host_in = {n: getattr(step, n).cpu().pin_memory() for n in names}
    host_out = [torch.empty_like(step.out, device="cpu").pin_memory() for _ in range(2)]
    dev = [{n: torch.empty_like(getattr(step, n)) for n in names + ("out",)} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = host_out[0].numel() * host_out[0].element_size()
    comp, cp = torch.cuda.current_stream(), torch.cuda.Stream()
    ready = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(cp):
        for n in names:
            dev[0][n].copy_(host_in[n], non_blocking=True)
        ready[0].record(cp)
    for i in range(steps):
        c, nx = i % 2, (i + 1) % 2
        comp.wait_event(ready[c])
        step.run(io=dev[c])
        done[c].record(comp)
        with torch.cuda.stream(cp):
            if i + 1 < steps:
                if i >= 1:
                    cp.wait_event(done[nx])     # step i-1 is done with the other set
                for n in names:
                    dev[nx][n].copy_(host_in[n], non_blocking=True)
                ready[nx].record(cp)
            cp.wait_event(done[c])
            host_out[c].copy_(dev[c]["out"], non_blocking=True)
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / steps
    return dt, h2d, d2h


def time_prefill_store(pkv, iters: int = 20):
    """kv_store of the varlen-prefill workload: 256 prompts, lengths U[100, 1024]."""
    lens = w.varlen_prefill_lengths()
    lay = w.varlen_prefill_layout(num_blocks=w.blocks_needed(lens) + 64)
    T = int(lens.sum())
    k = w.device_bf16_normal((T, HKV, D), 301)
    v = w.device_bf16_normal((T, HKV, D), 302)
    kc = torch.empty((lay.num_blocks, BS, HKV, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    slots = torch.from_numpy(lay.slot_mapping).cuda()
    for _ in range(3):
        pkv.kv_store(k, v, slots, kc, vc)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(iters):
        pkv.kv_store(k, v, slots, kc, vc)
    e1.record()
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3 / iters
    nbytes = 2 * T * ROW_BYTES * 2 + 8 * T
    del k, v, kc, vc
    return {"tokens": T, "gbs": nbytes / t / 1e9, "us": t * 1e6,
            "bytes": nbytes, "l2": "inputs (1.18 GB) larger than L2"}


def decode_shape_calls(pkv, batch: int, ctx: int):
    """`batch` sequences of `ctx` tokens (blocks drawn at random). Small batches rotate over
    enough disjoint copies of the pool region that the reads (>= 1 GB across the rotation)
    do not come from L2. Returns (call, reps, tables, keep): call(r) runs paged decode on
    copy r of reps; keep holds the device tensors alive."""
    per = batch * (-(-ctx // BS))
    reps = max(1, -(-(1 << 30) // (per * BS * ROW_BYTES * 2)))
    lay = w.decode_layout(np.full(batch * reps, ctx, np.int32), per * reps + 8, w.rng(5 + batch))
    kc = w.device_bf16_normal((lay.num_blocks, BS, HKV, D), 601)
    vc = w.device_bf16_normal((lay.num_blocks, BS, HKV, D), 602)
    q = w.device_bf16_normal((batch, HQ, D), 603)
    out = torch.empty_like(q)
    tables = [torch.from_numpy(lay.block_tables[r * batch:(r + 1) * batch].copy()).cuda()
              for r in range(reps)]
    cl = torch.full((batch,), ctx, dtype=torch.int32, device="cuda")
    ws = pkv.decode_workspace(batch, HQ, HKV, D, ctx, 0)
    call = lambda r: pkv.paged_decode_attn(q, kc, vc, tables[r], cl, ctx, D ** -0.5,
                                           workspace=ws, out=out)
    return call, reps, tables, (kc, vc, q, out, cl, ws)


def capture_graph(call, reps: int):
    """One CUDA graph holding call(0) .. call(reps - 1), back to back."""
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for r in range(reps):
                call(r)
    torch.cuda.current_stream().wait_stream(s)
    return g


def time_decode_shape(pkv, batch: int, ctx: int, hbm_peak: float, iters: int = 20,
                      graph: bool = False):
    """Paged decode attention alone on `batch` sequences of `ctx` tokens (decode_shape_calls).
    With `graph`, one CUDA graph holds one call per pool copy and is replayed, so the time is
    the GPU's alone (no host call overhead between launches)."""
    call, reps, tables, keep = decode_shape_calls(pkv, batch, ctx)
    for r in range(min(reps, 3)):
        call(r)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if graph:
        g = capture_graph(call, reps)
        replays = max(1, -(-iters // reps))
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(replays):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        n = replays * reps
    else:
        torch.cuda.synchronize()
        e0.record()
        for i in range(iters):
            call(i % reps)
        e1.record()
        torch.cuda.synchronize()
        n = iters
    t = e0.elapsed_time(e1) / 1e3 / n
    nbytes = decode_bytes(np.full(batch, ctx), tables[0].shape[1])["decode"]
    del keep
    return {"batch": batch, "ctx": ctx, "us": t * 1e6, "gbs": nbytes / t / 1e9,
            "frac_of_hbm_peak": nbytes / t / 1e9 / hbm_peak, "kv_tokens_per_s": batch * ctx / t,
            "timing": "cuda graph replay" if graph else "eager calls"}


def time_prefix_prefill(pkv, iters: int = 10):
    """Prefix-cached prefill: 64 sequences sharing a 2048-token prefix (8 ref-counted blocks)
    plus private suffixes of U[256, 768] tokens; queries are the suffixes, keys are read
    through block_table from the pool; one layer timed."""
    lay = w.prefix_prefill_case_layout(num_blocks=8 + 64 * 3 + 32)
    kc = w.device_bf16_normal((lay.num_blocks, BS, HKV, D), 701)
    vc = w.device_bf16_normal((lay.num_blocks, BS, HKV, D), 702)
    Tq = int(lay.seqlens_q.sum())
    q = w.device_bf16_normal((Tq, HQ, D), 703)
    out = torch.empty_like(q)
    cq = torch.from_numpy(lay.cu_seqlens_q).cuda()
    ck = torch.from_numpy(lay.cu_seqlens_k).cuda()
    bt = torch.from_numpy(lay.block_table).cuda()
    mq, mk = int(lay.seqlens_q.max()), int(lay.seqlens_k.max())
    call = lambda: pkv.varlen_prefill_attn(q, kc, vc, cq, ck, mq, mk, D ** -0.5, out=out,
                                           block_table=bt)
    for _ in range(3):
        call()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(iters):
        call()
    e1.record()
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3 / iters
    Lq = lay.seqlens_q.astype(np.int64)
    Lk = lay.seqlens_k.astype(np.int64)
    pairs = int((Lq * (Lk - Lq) + Lq * (Lq + 1) // 2).sum())
    flops = 4 * HQ * D * pairs
    return {"tflops": flops / t / 1e12, "ms": t * 1e3, "flops": flops, "causal_pairs": pairs,
            "query_tokens": Tq, "seqs": int(lay.n),
            "l2": "the 8 shared prefix blocks (8 MiB of K+V) stay in L2 across sequences"}


def time_qk_norm_rope_store(pkv, hbm_peak: float, iters: int = 20):
    """QK RMSNorm + RoPE fused into the store, on the varlen prefill workload's new tokens
    (145k tokens, positions within their prompts, the workload's slots)."""
    lens = w.varlen_prefill_lengths()
    lay = w.varlen_prefill_layout(num_blocks=w.blocks_needed(lens) + 64)
    T = int(lens.sum())
    g = w.rng(9)
    qkv = w.device_bf16_normal((T, (HQ + 2 * HKV) * D), 901)
    qw = torch.from_numpy(w.f32_to_bf16_bits(g.normal(1.0, 0.2, D).astype(np.float32))
                          .view(np.int16)).view(torch.bfloat16).cuda()
    kw = qw.clone()
    table = torch.from_numpy(w.random_cos_sin_table(g, 1024, D)).cuda()
    pos = torch.from_numpy(np.concatenate([np.arange(L) for L in lens]).astype(np.int64)).cuda()
    slots = torch.from_numpy(lay.slot_mapping).cuda()
    kc = torch.empty((lay.num_blocks, BS, HKV, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    q = torch.empty((T, HQ, D), dtype=torch.bfloat16, device="cuda")
    call = lambda: pkv.qk_norm_rope_store(qkv, pos, qw, kw, 1e-6, table, slots, kc, vc, HQ, HKV,
                                          q_out=q)
    for _ in range(3):
        call()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(iters):
        call()
    e1.record()
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3 / iters
    # projection rows in; q rows, K and V rows out; positions and slots
    nbytes = T * ((HQ + 2 * HKV) * D * 2 + HQ * D * 2 + 2 * HKV * D * 2 + 16)
    return {"tokens": T, "us": t * 1e6, "gbs": nbytes / t / 1e9, "bytes": nbytes,
            "frac_of_hbm_peak": nbytes / t / 1e9 / hbm_peak,
            "l2": "inputs (2.4 GB) larger than L2"}


def time_prefill(pkv, iters: int = 10, lens=None):
    """Varlen causal prefill attention: 256 prompts, lengths U[100, 1024], packed layout;
    one layer timed (x28 for a model). `lens` replaces the prompt lengths."""
    lens = w.varlen_prefill_lengths() if lens is None else np.asarray(lens, np.int32)
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).cuda()
    T = int(lens.sum())
    q = w.device_bf16_normal((T, HQ, D), 401)
    k = w.device_bf16_normal((T, HKV, D), 402)
    v = w.device_bf16_normal((T, HKV, D), 403)
    out = torch.empty_like(q)
    mx = int(lens.max())
    try:
        pkv.varlen_prefill_attn(q, k, v, cu, cu, mx, mx, D ** -0.5, out=out)
    except pkv.PkvError as e:
        return {"unavailable": str(e)}
    for _ in range(2):
        pkv.varlen_prefill_attn(q, k, v, cu, cu, mx, mx, D ** -0.5, out=out)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(iters):
        pkv.varlen_prefill_attn(q, k, v, cu, cu, mx, mx, D ** -0.5, out=out)
    e1.record()
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3 / iters
    pairs = int((lens.astype(np.int64) * (lens + 1) // 2).sum())
    flops = 4 * HQ * D * pairs
    return {"tflops": flops / t / 1e12, "ms": t * 1e3, "flops": flops, "causal_pairs": pairs}


def oracle_decode_sample(step: DecodeStep | None, seqs: int | None, layer: int = 0):
    """Inputs of one layer for the CPU oracle: referenced blocks copied to a compact host
    pool (untimed)."""
    import oracle  # CPU baseline only
    lay = step.lay
    rows = np.arange(lay.batch if seqs is None else seqs)
    tabs = lay.block_tables[rows]
    ids = np.unique(tabs[tabs >= 0])
    remap = np.full(lay.num_blocks, -1, np.int64)
    remap[ids] = np.arange(len(ids))
    idt = torch.from_numpy(ids).long().cuda()

    def bits(t):
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

    kc = bits(step.pool[0, layer][idt])
    vc = bits(step.pool[1, layer][idt])
    bt = np.where(tabs >= 0, remap[np.maximum(tabs, 0)], -1).astype(np.int32)
    slots_blk = remap[lay.slot_mapping[rows] // BS] * BS + lay.slot_mapping[rows] % BS
    return dict(oracle=oracle, q=bits(step.q[layer])[rows], kn=bits(step.kn[layer])[rows],
                vn=bits(step.vn[layer])[rows], kc=kc, vc=vc, bt=bt,
                ctx=lay.context_lens[rows], slots=slots_blk.astype(np.int64),
                bytes=decode_bytes(lay.context_lens[rows], lay.block_tables.shape[1]))


def oracle_step_time(s, num_threads: int = 0) -> float:
    o = s["oracle"]
    t0 = time.perf_counter()
    o.kv_store(s["kn"], s["vn"], s["slots"], s["kc"], s["vc"])
    o.paged_decode(s["q"], s["kc"], s["vc"], s["bt"], s["ctx"], D ** -0.5,
                   num_threads=num_threads)
    return time.perf_counter() - t0


# ------------------------------------------------------------------------------- arms
def load_pkv():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_pkv_build", os.path.join(ROOT, "paged_kv_cache_208_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    import paged_kv_cache_208_gb300 as pkv
    return pkv


def run_ours(args):
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl")
    pkv = load_pkv()
    hbm_peak, bf16_peak, bf16_sus, peak_src = peaks()

    step = DecodeStep(pkv, pool_fraction=args.pool_fraction, rank=rank, world=world,
                      num_splits=args.num_splits)
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    if pkv.get_device_errors():
        raise RuntimeError("device error bits set during warm-up")

    with ClockSampler(torch.cuda.current_device()) as clocks:
        # timed region 1: the headline, blocks of exactly K steps back to back, each bracketed
        # by a barrier and a synchronize; blocks repeat until they cover MIN_TIMED_SECONDS so
        # that the clock sampler sees the GPU under load (value: the median block)
        block_times, covered = [], 0.0
        while covered < MIN_TIMED_SECONDS or not block_times:
            barrier(world)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(args.steps):
                step.run()
            e1.record()
            torch.cuda.synchronize()
            barrier(world)
            block_times.append(max_over_ranks(e0.elapsed_time(e1) / 1e3, world))
            covered += block_times[-1]
            if len(block_times) >= 1000:
                break
        # timed region 2: K steps with an event pair around every decode call, for the decode
        # kernel's own launch duration (roofline)
        events = []
        for _ in range(args.steps):
            step.run(events)
        torch.cuda.synchronize()
    elapsed = statistics.median(block_times)
    per_step = elapsed / args.steps
    decode_times = [a.elapsed_time(b) / 1e3 for a, b in zip(events[0::2], events[1::2])]
    decode_avg = sum(decode_times) / len(decode_times)

    e2e_dt, h2d, d2h = time_e2e(step, min(args.steps, 50))
    e2e_dt = max_over_ranks(e2e_dt, world)

    extra = {}
    if not args.skip_extra:
        extra["decode_long_context"] = time_decode_shape(pkv, 32, 32768, hbm_peak)
        keep = ("batch", "us", "gbs", "frac_of_hbm_peak")
        extra["decode_batch_sweep"] = {
            "ctx": 1024, "timing": "CUDA graph replay of back-to-back calls",
            "points": [{k: v for k, v in time_decode_shape(pkv, b, 1024, hbm_peak,
                                                           graph=True).items() if k in keep}
                       for b in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512)]}
        extra["decode_batch_sweep"]["first_batch_at_70pct"] = next(
            (p["batch"] for p in extra["decode_batch_sweep"]["points"]
             if p["frac_of_hbm_peak"] >= 0.7), None)
        extra["decode_batch_sweep_eager"] = [
            {k: v for k, v in time_decode_shape(pkv, b, 1024, hbm_peak).items() if k in keep}
            for b in (1, 8, 64)]
        extra["kv_store_prefill"] = time_prefill_store(pkv)
        extra["qk_norm_rope_store_prefill"] = time_qk_norm_rope_store(pkv, hbm_peak)
        extra["prefill"] = time_prefill(pkv)
        if "tflops" in extra["prefill"]:
            extra["prefill"]["frac_of_bf16_peak"] = extra["prefill"]["tflops"] / bf16_peak
            extra["prefill"]["tflops_x28_layers_ms"] = extra["prefill"]["ms"] * LAYERS
        # the same kernel on long prompts (16 x 8192 tokens): few item switches and diagonal
        # tiles, so this is its steady-state rate, beside the short prompts above
        extra["prefill_long_prompts"] = time_prefill(pkv, iters=5, lens=[8192] * 16)
        if "tflops" in extra["prefill_long_prompts"]:
            extra["prefill_long_prompts"]["frac_of_bf16_peak"] = (
                extra["prefill_long_prompts"]["tflops"] / bf16_peak)
            extra["prefill_long_prompts"]["prompts"] = "16 x 8192 tokens, causal, packed"
        extra["prefix_prefill"] = time_prefix_prefill(pkv)
        extra["prefix_prefill"]["frac_of_bf16_peak"] = extra["prefix_prefill"]["tflops"] / bf16_peak

    cpu = None
    if rank == 0 and not args.skip_cpu:
        s = oracle_decode_sample(step, None)
        import oracle
        # repeat one layer's work until about 10 s of CPU time have run (each repeat writes
        # the same rows, so the inputs do not change between repeats)
        reps, total = 0, 0.0
        while total < 10.0 and reps < 1000:
            total += oracle_step_time(s)
            reps += 1
        t = total / reps
        nbytes = s["bytes"]["store"] + s["bytes"]["decode"]
        # the same layer on one thread, a few repeats
        reps1, total1 = 0, 0.0
        while total1 < 3.0 and reps1 < 100:
            total1 += oracle_step_time(s, num_threads=1)
            reps1 += 1
        cpu = {"value": nbytes / t / 1e9, "unit": "GB/s",
               "cores": oracle.max_threads(), "kind": "oracle",
               "sample": f"one layer (of 28) of the full batch, repeated {reps} times: kv_store "
                         "+ paged decode of all 256 sequences, fp64 C oracle with OpenMP",
               "seconds": total,
               "one_thread": {"value": nbytes / (total1 / reps1) / 1e9, "unit": "GB/s",
                              "repeats": reps1, "seconds": total1}}
    if rank != 0:
        return
    total_bytes = step.step_bytes * world
    dec_bytes = step.bytes["decode"] + step.bytes["store"]  # the call stores and attends
    traffic, traffic_note = decode_traffic()
    achieved = dec_bytes / decode_avg / 1e9
    line = {
        "metric": METRIC,
        "value": total_bytes / per_step / 1e9,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": per_step * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, seeded lengths and block draws)",
        "config": {"workload": WORKLOAD, "batch": step.B, "layers": LAYERS,
                   "sum_ctx": int(step.lay.context_lens.sum()), "num_blocks": step.num_blocks,
                   "pool_gb": round(step.pool.numel() * 2 / 1e9, 1),
                   "splits": args.num_splits or "auto", "l2": "inputs larger than L2 (1.13 GB of KV per layer)",
                   "timed_blocks": len(block_times), "timed_seconds": round(covered, 3),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "kv_tokens_per_s": step.kv_tokens * world / per_step,
        "decode_frac_of_hbm_peak": achieved / hbm_peak,
        "roofline": {"bound": "hbm",
                     "kernel": "paged_decode_step (split kernel with the store; + the merge kernel when contexts are split)",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "peak_source": peak_src,
                     "traffic": traffic,
                     "traffic_kernel": "decode_split_kernel (ncu, one launch, same workload)",
                     "traffic_source": traffic_note,
                     "algorithmic_bytes_per_launch": dec_bytes,
                     "avg_launch_us": decode_avg * 1e6},
        "e2e": {"value": total_bytes / e2e_dt / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_dt * 1e3,
                "copies": "pinned host <-> device every step, on a second stream overlapping "
                          "the neighbouring steps' compute (two device buffer sets)"},
        "gpu_launches": step.launches_per_step() * args.steps,
        "gpu_launches_counted_over": "one timed block of K steps",
        "clocks": clocks.summary(),
        "cpu_baseline": cpu,
        "extra": extra,
    }
    print(json.dumps(line), flush=True)


def reference_inputs(seqs: int = 16, seed: int = 2):
    """Inputs of one layer of the decode step for the reference arm, made on the host alone:
    the first `seqs` sequences of the Qwen3 decode batch (their lengths, block draws and new
    tokens' slots), a compact pool of just the blocks they reference, and bf16 N(0,1) values
    drawn with numpy. No device memory and no part of the CUDA library are involved."""
    import oracle  # the reference arm times the oracle
    ctx_all = w.qwen3_decode_lengths(seed)
    lay = w.qwen3_decode_layout(w.blocks_needed(ctx_all) + 64, seed)
    rows = np.arange(seqs)
    tabs = lay.block_tables[rows]
    ids = np.unique(tabs[tabs >= 0])
    remap = np.full(lay.num_blocks, -1, np.int64)
    remap[ids] = np.arange(len(ids))
    bt = np.where(tabs >= 0, remap[np.maximum(tabs, 0)], -1).astype(np.int32)
    slots = remap[lay.slot_mapping[rows] // BS] * BS + lay.slot_mapping[rows] % BS
    g = w.rng(10_000 + seed)
    return dict(oracle=oracle, q=w.host_bf16_normal(g, (seqs, HQ, D)),
                kn=w.host_bf16_normal(g, (seqs, HKV, D)), vn=w.host_bf16_normal(g, (seqs, HKV, D)),
                kc=w.host_bf16_normal(g, (len(ids), BS, HKV, D)),
                vc=w.host_bf16_normal(g, (len(ids), BS, HKV, D)), bt=bt,
                ctx=lay.context_lens[rows], slots=slots.astype(np.int64),
                bytes=decode_bytes(lay.context_lens[rows], lay.block_tables.shape[1]))


def run_reference(args):
    """The CPU oracle timed on the host cores, on the same workload and metric: each step is a
    bounded sample (16 of the 256 sequences of one layer: store + paged decode). Its inputs are
    made on the host (reference_inputs): this arm loads no part of the CUDA library."""
    rank, world, local = dist_env()
    if rank != 0:
        return
    s = reference_inputs(16)
    oracle = s["oracle"]
    base_kc, base_vc = s["kc"].copy(), s["vc"].copy()
    times = []
    for i in range(args.warmup + args.steps):
        s["kc"], s["vc"] = base_kc.copy(), base_vc.copy()
        t = oracle_step_time(s)
        if i >= args.warmup:
            times.append(t)
    per = sum(times) / len(times)
    nbytes = s["bytes"]["store"] + s["bytes"]["decode"]
    value = nbytes / per / 1e9
    sample = ("16 of the 256 sequences of one layer per step: kv_store + paged decode, "
              "fp64 C oracle with OpenMP, inputs drawn on the host")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same seeded workload shape: lengths, block draws, slots)",
        "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def run_profile(args):
    """One kernel alone on its workload, for ncu: `decode` (the Qwen3 batch, one layer, a pool
    of just the referenced blocks: 1.2 GB, larger than L2), `decode_small` (--profile-batch
    sequences of 1024 tokens, graph-replayed), `decode_long` (8 x 32768), `prefill` (the varlen workload,
    packed), `prefill_long` (16 prompts of 8192 tokens, packed), `prefix` (the prefix-cached
    workload, keys through block_table) or `store` (the varlen workload's kv_store). Runs
    --warmup + --steps launches."""
    torch.cuda.set_device(0)
    pkv = load_pkv()
    if args.profile == "decode":
        ctx = w.qwen3_decode_lengths()
        step = DecodeStep(pkv, num_blocks=w.blocks_needed(ctx) + 8, layers=1,
                          num_splits=args.num_splits)
        s = step.pool
        run = lambda: pkv.paged_decode_step(step.q[0], step.kn[0], step.vn[0], step.slots,
                                            s[0, 0], s[1, 0], step.tables, step.ctx, step.maxc,
                                            step.lay.scale, num_splits=args.num_splits,
                                            workspace=step.ws, out=step.out[0])
    elif args.profile == "decode_small":
        # --profile-batch sequences of 1024 tokens through the batch sweep's rotation of pool
        # copies; one CUDA graph of one call per copy, replayed (--warmup + --steps) times
        call, reps, _, keep = decode_shape_calls(pkv, args.profile_batch, 1024)
        g = capture_graph(call, reps)
        run = g.replay
    elif args.profile == "decode_long":
        # the long-context shape reduced to 8 sequences x 32768 tokens (1.07 GB of K+V)
        call, reps, _, keep = decode_shape_calls(pkv, 8, 32768)
        run = lambda: call(0)
    elif args.profile == "store":
        lens = w.varlen_prefill_lengths()
        lay = w.varlen_prefill_layout(num_blocks=w.blocks_needed(lens) + 64)
        T = int(lens.sum())
        k, v = (w.device_bf16_normal((T, HKV, D), 301 + i) for i in range(2))
        kc = torch.empty((lay.num_blocks, BS, HKV, D), dtype=torch.bfloat16, device="cuda")
        vc = torch.empty_like(kc)
        slots = torch.from_numpy(lay.slot_mapping).cuda()
        run = lambda: pkv.kv_store(k, v, slots, kc, vc)
    elif args.profile == "rope":
        lens = w.varlen_prefill_lengths()
        lay = w.varlen_prefill_layout(num_blocks=w.blocks_needed(lens) + 64)
        T = int(lens.sum())
        qkv = w.device_bf16_normal((T, (HQ + 2 * HKV) * D), 901)
        qw = torch.ones(D, dtype=torch.bfloat16, device="cuda")
        table = torch.from_numpy(w.random_cos_sin_table(w.rng(9), 1024, D)).cuda()
        pos = torch.from_numpy(np.concatenate([np.arange(L) for L in lens]).astype(np.int64)).cuda()
        slots = torch.from_numpy(lay.slot_mapping).cuda()
        kc = torch.empty((lay.num_blocks, BS, HKV, D), dtype=torch.bfloat16, device="cuda")
        vc = torch.empty_like(kc)
        run = lambda: pkv.qk_norm_rope_store(qkv, pos, qw, qw, 1e-6, table, slots, kc, vc, HQ, HKV)
    elif args.profile == "prefix":
        lay = w.prefix_prefill_case_layout(num_blocks=8 + 64 * 3 + 32)
        kc = w.device_bf16_normal((lay.num_blocks, BS, HKV, D), 701)
        vc = w.device_bf16_normal((lay.num_blocks, BS, HKV, D), 702)
        q = w.device_bf16_normal((int(lay.seqlens_q.sum()), HQ, D), 703)
        out = torch.empty_like(q)
        cq = torch.from_numpy(lay.cu_seqlens_q).cuda()
        ck = torch.from_numpy(lay.cu_seqlens_k).cuda()
        bt = torch.from_numpy(lay.block_table).cuda()
        mq, mk = int(lay.seqlens_q.max()), int(lay.seqlens_k.max())
        run = lambda: pkv.varlen_prefill_attn(q, kc, vc, cq, ck, mq, mk, D ** -0.5, out=out,
                                              block_table=bt)
    else:
        lens = (np.full(16, 8192, np.int32) if args.profile == "prefill_long"
                else w.varlen_prefill_lengths())
        cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).cuda()
        T = int(lens.sum())
        q = w.device_bf16_normal((T, HQ, D), 401)
        k = w.device_bf16_normal((T, HKV, D), 402)
        v = w.device_bf16_normal((T, HKV, D), 403)
        out = torch.empty_like(q)
        mx = int(lens.max())
        run = lambda: pkv.varlen_prefill_attn(q, k, v, cu, cu, mx, mx, D ** -0.5, out=out)
    for _ in range(args.warmup + args.steps):
        run()
    torch.cuda.synchronize()
    errors = pkv.get_device_errors()
    print(json.dumps({"profile": args.profile, "launches": args.warmup + args.steps,
                      "device_errors": errors}))
    if errors:
        sys.exit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--pool-fraction", type=float, default=0.9,
                    help="fraction of free HBM for the KV pool (the workload says 0.9)")
    ap.add_argument("--skip-extra", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--num-splits", type=int, default=0,
                    help="decode KV splits of the longest context (0 = the library's choice)")
    ap.add_argument("--profile-batch", type=int, default=8,
                    help="sequences for --profile decode_small")
    ap.add_argument("--profile", choices=["decode", "decode_small", "decode_long", "prefill",
                                          "prefill_long", "prefix", "store", "rope"],
                    help="run one kernel alone (for ncu); prints no benchmark line")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile:
        run_profile(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
