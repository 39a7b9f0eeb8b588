"""Benchmark of the tree-training hot path on GB300.

One step = one pass of every device row of the path over one synthetic
workload (``--config``, default 2):
    block classification -> tree attention forward -> tree attention backward
    [-> log-softmax / entropy / label gather -> per-sequence regather]
Config 2 (the default, the headline line) is the GRPO-shaped workload
(8 prompts x 8 samples, bimodal responses, max_tokens_per_mb 8192, 32 query /
8 kv heads, head_dim 128) with its log-prob pass over bf16 logits of width
151936 on the same packed trees (the log-prob workload).  Config 1 (tiny,
with log-probs over a 1000-wide vocabulary), config 3 (agentic multi-turn,
one deep tree) and config 5 (64K-token few-shot tree) time their attention
forward and backward; configs 3 and 5 name no logits.
The packed metadata and every input are resident in HBM when the timed
region starts (``value``); ``e2e`` repeats the step through the public API
from host buffers: host packing, metadata upload, host->device copies of
q, k, v, dO (and logits) from pinned memory, the device work, and the
device->host copies of O, dQ, dK, dV (and the per-sequence log-probs and
entropies).

Metric: ancestor-pair attention FLOPs (FlashAttention convention, forward
4 P d Hq, backward 2.5x, i.e. 14 P d Hq per step, P = sum of depth + 1 over
tree tokens) per second of the whole step; tree tokens/s is reported beside
it, and the strict count without the recomputed S (12 P d Hq).  Inputs of
configs 2, 3 and 5 (q alone is 470 MB to 4.3 GB) are larger than the 129 MB
L2, so no flush is needed between their steps; config 1 writes a 256 MB
buffer between steps to flush the L2.

``--impl reference`` times the CPU oracle (fp64, host cores) on a bounded
sample of the same workload and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "tree-attn fwd+bwd TFLOP/s on ancestor pairs (% bf16 peak); tree tokens/s"
UNIT = "TFLOP/s"
WORKLOADS = {
    1: ("Tiny tree-attn: 4 prompts x 4 samples, prompt 64 tokens, responses 16-64 tokens, vocab 1000, "
        "max_tokens_per_mb 1024, 4 q / 4 kv heads, head_dim 64, bf16; log-probs over bf16 logits "
        "[tree tokens, 1000]"),
    2: ("GRPO-shaped: 8 prompts x 8 samples, prompts 256-1024, responses 70% 50-200 / 30% 800-2048 "
        "tokens, vocab 32000, max_tokens_per_mb 8192, 32 q / 8 kv heads, head_dim 128, bf16; "
        "log-probs over bf16 logits [tree tokens, 151936] on the same trees"),
    3: ("Agentic multi-turn: shared 2048-token system prompt, 16 trajectories of 4-8 turns of 64-512 "
        "tokens, branch factor 1-3, max_tokens_per_mb 32768, 16 q / 2 kv heads, head_dim 128, bf16 "
        "fwd+bwd"),
    5: ("Large few-shot tree: shared 4096-token prefix, 64 samples of 512-4096 tokens branching at up to "
        "16 depths, max_tokens_per_mb 65536, 32 q / 8 kv heads, head_dim 128, bf16 fwd+bwd"),
}
WORKLOAD = WORKLOADS[2]
NOMINAL_HBM_GBS = 8000.0   # the HBM figure the log-prob target is stated against
# A timed region shorter than this runs at the burst clock; longer ones at the
# clock the power cap settles to.
SUSTAINED_AFTER_S = 1.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


# Per-launch DRAM traffic comes from the ncu summaries under profiles/: each
# names the source file it was captured from and that file's sha256 prefix,
# the tree tokens of the captured case, and "DRAM traffic (read + write) of
# this launch: X GB".  A summary counts only while the source is unchanged;
# attention and log-prob traffic scale with the tree tokens processed (every
# Q, K, V, O, dO, gradient and logits row is read or written a fixed number
# of times).  The summaries were taken on the GRPO-shaped workload (config 2).
PROFILES = {
    "tpa_tree_attn_fwd": ["attn_fwd_grpo_3trees_ncu_full.md"],
    "tpa_tree_attn_bwd": ["bwd_pre_grpo_3trees_ncu_full.md", "attn_bwd_kv_grpo_3trees_ncu_full.md",
                          "attn_bwd_dq2_grpo_3trees_ncu_full.md"],
    "tpa_tree_logprobs_entropy": ["logprobs_row_grpo_1tree_ncu.md"],
}


def _profile_traffic(entry: str, tree_tokens: int):
    import hashlib
    import re
    total = 0.0
    for name in PROFILES.get(entry, []):
        path = os.path.join(ROOT, "profiles", name)
        if not os.path.exists(path):
            return None
        text = open(path).read()
        src = re.search(r"Source: `([^`]+)` sha256 prefix ([0-9a-f]+)", text)
        gb = re.search(r"DRAM traffic \(read \+ write\) of this launch: ([0-9.]+) GB", text)
        toks = re.search(r"\(([0-9]+) tree tokens", text)
        if not (src and gb and toks):
            return None
        with open(os.path.join(ROOT, src.group(1)), "rb") as f:
            if not hashlib.sha256(f.read()).hexdigest().startswith(src.group(2)):
                return None  # the kernel changed since the counters were taken
        total += float(gb.group(1)) * 1e9 * tree_tokens / int(toks.group(1))
    return total if total > 0 else None


def rank_sequences(rank: int, world: int, tpa, cid: int = 2):
    """The sequences rank ``rank`` of ``world`` processes.

    One rank: the workload's batch (seed = config id).  N ranks: N such
    batches (seeds cid + 1000 r) are packed together on every rank (the packer
    is deterministic), and the trees are split over the ranks by KK balancing
    of each tree's ancestor pairs, the attention work; a rank keeps the
    sequences of its trees.  Per-rank work stays that of one batch (weak
    scaling) and the data path needs no collective."""
    from synth import CONFIGS, flatten_sequences, make_sequences
    if world == 1:
        return make_sequences(cid, seed=cid)
    seqs = [s for r in range(world) for s in make_sequences(cid, seed=cid + 1000 * r)]
    toks, offs = flatten_sequences(seqs)
    tree = tpa.tree_pack(tokens=toks, offsets=offs, max_tokens_per_mb=CONFIGS[cid].max_tokens_per_mb)
    arr = tree.arrays()
    depth, ntok = arr["depth"].reshape(tree.n_trees, -1), arr["n_tokens"]
    pairs = [int((depth[b, :ntok[b]] + 1).sum()) for b in range(tree.n_trees)]
    group_of, n_groups, _ = tpa.balance(pairs, 10**15, world, 1, "kk")
    mine = {b for b in range(tree.n_trees) if group_of[b] == rank % n_groups}
    return [s for s, b in zip(seqs, arr["seq_tree"]) if int(b) in mine]


def reduce_job(flops: float, rows: int, ms: float):
    """Whole-job totals over the ranks: work summed, time the slowest rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return flops, rows, ms
    t = torch.tensor([flops, float(rows)], dtype=torch.float64)
    m = torch.tensor([ms], dtype=torch.float64)
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t, m = t.to(dev), m.to(dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    dist.all_reduce(m, op=dist.ReduceOp.MAX)
    return float(t[0]), int(t[1]), float(m[0])


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *a):
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
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def segment_stats(seg):
    """Median and spread (min, p10, p90, max) of per-step segment times [ms]."""
    import numpy as np
    seg = np.asarray(seg, dtype=np.float64)
    return {"median": float(np.median(seg)), "min": float(seg.min()), "p10": float(np.percentile(seg, 10)),
            "p90": float(np.percentile(seg, 90)), "max": float(seg.max())}


def pick_bf16_peak(peaks: dict, timed_s: float):
    """The bf16 denominator for a kernel timed inside a region of ``timed_s``
    seconds: the burst figure below SUSTAINED_AFTER_S, the sustained one above."""
    if timed_s < SUSTAINED_AFTER_S or "bf16_tflops_sustained" not in peaks:
        return peaks["bf16_tflops"], "bf16 burst"
    return peaks["bf16_tflops_sustained"], "bf16 sustained"


# ---------------------------------------------------------------- CPU oracle (reference arm / cpu_baseline)

def _oracle_sample(cfg, seqs, budget_pairs: int):
    """Nodes of tree 0 (shortest first) whose ancestor pairs sum to about
    ``budget_pairs``; returns (packing, tree, nodes, pairs)."""
    import numpy as np
    import oracle
    pk = oracle.tree_pack(seqs, cfg.max_tokens_per_mb)
    t = pk.trees[0]
    order = np.argsort(t.node_end - t.node_start, kind="stable")
    nodes, pairs = [], 0
    for nid in order:
        s0, s1 = int(t.node_start[nid]), int(t.node_end[nid])
        p = int((t.depth[s0:s1 + 1] + 1).sum())
        if pairs + p > budget_pairs and nodes:
            continue
        nodes.append(int(nid))
        pairs += p
        if pairs >= budget_pairs:
            break
    return pk, t, nodes, pairs


def _oracle_step(cfg, t, nodes, q, k, v, do):
    import oracle
    oracle.attn_forward(t, q, k, v, t_pad=cfg.max_tokens_per_mb, nodes=nodes)
    oracle.attn_backward(t, q, k, v, do, t_pad=cfg.max_tokens_per_mb, nodes=nodes)


def cpu_oracle_run(steps: int, warmup: int, budget_pairs: int, cid: int = 2):
    """Time the fp64 oracle's attention fwd+bwd on a bounded sample."""
    import torch
    from synth import CONFIGS, make_sequences
    cfg = CONFIGS[cid]
    seqs = make_sequences(cid)
    pk, t, nodes, pairs = _oracle_sample(cfg, seqs, budget_pairs)
    T = cfg.max_tokens_per_mb
    g = torch.Generator().manual_seed(1000 * cid + 1)
    q = torch.randn((T, cfg.n_heads_q, cfg.head_dim), generator=g).to(torch.bfloat16)
    k = torch.randn((T, cfg.n_heads_kv, cfg.head_dim), generator=g).to(torch.bfloat16)
    v = torch.randn((T, cfg.n_heads_kv, cfg.head_dim), generator=g).to(torch.bfloat16)
    do = torch.randn((T, cfg.n_heads_q, cfg.head_dim), generator=g).to(torch.bfloat16)
    for _ in range(warmup):
        _oracle_step(cfg, t, nodes, q, k, v, do)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        _oracle_step(cfg, t, nodes, q, k, v, do)
        times.append(time.perf_counter() - t0)
    flops = 14.0 * pairs * cfg.head_dim * cfg.n_heads_q
    sec = sum(times) / len(times)
    whole = pairs == int((t.depth[:t.n] + 1).sum()) and pk.n_trees == 1
    sample = (f"oracle fp64 attention fwd+bwd on {len(nodes)} nodes of tree 0 "
              f"({'the whole workload' if whole else 'shortest first'}), "
              f"{pairs} ancestor pairs x {cfg.n_heads_q} heads x d {cfg.head_dim}; "
              f"{sec:.2f} s per step")
    return {"value": flops / sec / 1e12, "sec_per_step": sec, "pairs": pairs, "nodes": len(nodes),
            "sample": sample, "cores": torch.get_num_threads(), "tree_tokens_per_s":
            sum(int(t.node_end[n] - t.node_start[n] + 1) for n in nodes) / sec}


def cpu_oracle_side(cid: int, logits_vocab: int | None, n_rows: int = 64):
    """The oracle packer on the whole workload, and the oracle log-prob pass
    on ``n_rows`` tree rows (fp64 log-softmax + entropy + label gather)."""
    import numpy as np
    import torch
    import oracle
    from synth import CONFIGS, make_sequences
    cfg = CONFIGS[cid]
    seqs = make_sequences(cid)
    t0 = time.perf_counter()
    pk = oracle.tree_pack(seqs, cfg.max_tokens_per_mb)
    pack_s = time.perf_counter() - t0
    out = {"pack_s": pack_s, "pack_tokens_per_s": pk.total_seq_tokens / pack_s,
           "pack_sample": f"oracle packer on the whole workload ({len(seqs)} sequences, "
                          f"{pk.total_seq_tokens} tokens)"}
    if logits_vocab:
        t = pk.trees[0]
        rows = min(n_rows, t.n)
        logits = (2 * torch.randn((rows, logits_vocab), generator=torch.Generator().manual_seed(5))
                  ).to(torch.bfloat16)
        pos = list(range(rows))
        t0 = time.perf_counter()
        oracle.position_logprobs_entropy(pk, logits, [0] + [0] * (pk.n_trees - 1), 0,
                                         [p for p in pos if t.parent[p] < rows])
        lp_s = time.perf_counter() - t0
        nbytes = rows * logits_vocab * 2
        out.update({"logprobs_s": lp_s, "logprobs_gbs": nbytes / lp_s / 1e9,
                    "logprobs_sample": f"oracle fp64 log-prob pass on {rows} tree rows x {logits_vocab}"})
    return out


def reference_budget(oracle_pairs: int, steps: int, warmup: int) -> int:
    """Ancestor pairs of each reference step's sample: it shrinks with the
    number of steps, so that a whole --steps K --warmup W run stays near
    twelve full-size samples (a few minutes on the host cores)."""
    n = max(1, steps + warmup)
    return max(1, int(oracle_pairs * min(1.0, 12.0 / n)))


def run_reference(args, rank, world):
    if rank != 0:
        return
    r = cpu_oracle_run(args.steps, args.warmup, reference_budget(args.oracle_pairs, args.steps, args.warmup),
                       args.config)
    line = {
        "impl": "reference", "metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["sec_per_step"] * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOADS[args.config], "sample": "bounded oracle sample"},
        "cpu_baseline": {"value": r["value"], "unit": UNIT, "cores": r["cores"], "kind": "oracle",
                         "sample": r["sample"]},
        "e2e": {"value": r["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm

def run_gpu(args, rank, world, local):
    import numpy as np
    import torch
    import torch.distributed as dist

    import prefix_shared_tree_attention_gb300 as tpa
    from synth import (CONFIGS, flatten_sequences, make_dout, make_hidden, make_lm_weight, make_logits, make_qkv,
                       make_sequences)

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    tpa.device_check()
    cid = args.config
    cfg = CONFIGS[cid]
    # logits of the log-prob pass: config 2 uses the log-prob workload (its
    # trees, width 151936, seed 4); config 1 its own 1000-wide logits
    lp_cid = {1: 1, 2: 4}.get(cid)
    seqs = rank_sequences(rank, world, tpa, cid)  # weak scaling: one batch's worth of trees per rank
    toks, offs = flatten_sequences(seqs)
    T, Hq, Hkv, d = cfg.max_tokens_per_mb, cfg.n_heads_q, cfg.n_heads_kv, cfg.head_dim
    V = CONFIGS[lp_cid].logits_vocab if lp_cid else 0

    tree = tpa.tree_pack(tokens=toks, offsets=offs, max_tokens_per_mb=T)
    if args.max_trees and tree.n_trees > args.max_trees:
        # profiling: keep only the sequences of the first trees and repack them
        keep = tree.arrays()["seq_tree"] < args.max_trees
        seqs = [s for s, kp in zip(seqs, keep) if kp]
        toks, offs = flatten_sequences(seqs)
        tree = tpa.tree_pack(tokens=toks, offsets=offs, max_tokens_per_mb=T)
    info = tree.info
    B = info.n_trees
    run_attn = args.only in ("all", "attn")
    run_lp = args.only in ("all", "logprobs") and lp_cid is not None
    rows = info.total_tree_tokens
    pairs = int(info.ancestor_pairs)
    flops_fwd = 4.0 * pairs * d * Hq
    flops_bwd = 10.0 * pairs * d * Hq
    flops_step = 14.0 * pairs * d * Hq if run_attn else 0.0
    flops_strict = 12.0 * pairs * d * Hq if run_attn else 0.0

    dtree = tree.upload(dev)
    mask = tpa.BlockMask(B, T, dev)
    qh, kh, vh = make_qkv(cid, B, T, Hq, Hkv, d)
    doh = make_dout(cid, B, T, Hq, d)
    q, k, v, do = (x.to(dev) for x in (qh, kh, vh, doh))
    logits = make_logits(lp_cid, rows, V, device=str(dev)) if run_lp else None
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device=dev)
    # gradients in the dtype the workload fixes (bf16, as q/k/v); --grad-dtype fp32 times the
    # fp32-output path, which splits long key columns into items that add into zeroed rows
    gdt = torch.float32 if args.grad_dtype == "fp32" else torch.bfloat16
    dq, dk, dv = (torch.empty(x.shape, dtype=gdt, device=dev) for x in (q, k, v))
    ws = torch.empty(tpa.tree_attn_bwd_workspace_bytes(B, T, Hq, Hkv, d, gdt), dtype=torch.uint8, device=dev)
    N = info.total_seq_tokens
    lp_out = (torch.empty((B, T), dtype=torch.float32, device=dev), torch.empty((B, T), dtype=torch.float32, device=dev),
              torch.empty(N, dtype=torch.float32, device=dev), torch.empty(N, dtype=torch.float32, device=dev))
    stream = torch.cuda.current_stream(dev)
    # inputs smaller than the L2 (config 1): flush it between steps, outside the segments
    in_bytes = sum(x.numel() * x.element_size() for x in (q, k, v, do)) + (
        logits.numel() * logits.element_size() if logits is not None else 0)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if in_bytes < (256 << 20) else None
    n_launch_per_step = 3 + (1 + 3 if run_attn else 0) + (2 if run_lp else 0)

    def step(ev=None):
        if flush is not None:
            flush.fill_(1)
        if ev: ev[0].record(stream)
        tpa.block_classify(dtree, out=mask)
        if ev: ev[1].record(stream)
        if run_attn:
            tpa.tree_attn_fwd(dtree, mask, q, k, v, out=o, lse=lse)
        if ev: ev[2].record(stream)
        if run_attn:
            tpa.tree_attn_bwd(dtree, mask, q, k, v, o, lse, do, workspace=ws, out=(dq, dk, dv), grad_dtype=gdt)
        if ev: ev[3].record(stream)
        if run_lp:
            tpa.tree_logprobs_entropy(dtree, logits, out=lp_out)
        if ev: ev[4].record(stream)

    for _ in range(args.warmup):
        step()
    tpa.sync_status()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    tpa.sync_status()
    total_ms = t_start.elapsed_time(t_end)
    seg = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(4)] for i in range(args.steps)])
    stats = {name: segment_stats(seg[:, j]) for j, name in
             enumerate(("block_classify", "attn_fwd", "attn_bwd", "logprobs_entropy"))}
    t_cls, t_fwd, t_bwd, t_lp = (stats[n]["median"] for n in
                                 ("block_classify", "attn_fwd", "attn_bwd", "logprobs_entropy"))
    # the step as a whole: the device time between the first and last events
    # (a flush between steps, when there is one, is not part of it)
    step_ms = np.array([evs[i][0].elapsed_time(evs[i][4]) for i in range(args.steps)])
    if flush is not None:
        total_ms = float(step_ms.sum())
    # whole job: work summed over the ranks, time of the slowest rank
    job_flops, job_rows, total_ms = reduce_job(flops_step, rows, total_ms)
    ms_step = total_ms / args.steps
    clocks = clk.summary()

    # ------------------------------------------------ dense ancestor-mask export (Megatron-style mask)
    # Not part of the step: the export a dense-mask consumer would run once
    # per micro-batch, timed alone on the same trees; bound by HBM writes.
    dmask = None
    if args.only in ("all", "attn") and not args.no_extras:
        dmask = {}
        for fmt in ("u8", "bits"):
            buf = tpa.dense_mask(dtree, fmt)
            for _ in range(3):
                tpa.dense_mask(dtree, fmt, out=buf)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = 10
            e0.record(stream)
            for _ in range(reps):
                tpa.dense_mask(dtree, fmt, out=buf)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ms = e0.elapsed_time(e1) / reps
            nbytes = buf.numel() * buf.element_size()
            dmask[fmt] = {"ms": ms, "bytes": nbytes, "gbs": nbytes / (ms / 1e3) / 1e9}
            del buf
        tpa.sync_status()

    peaks, peak_kind = _peaks()

    # ------------------------------------------------ LM head fused into the log-prob pass
    # The step upstream of the log-prob rows: logits = hidden @ W^T formed on
    # tcgen05 tiles and consumed in place.  Hidden size 4096 (a reading: the
    # pages give none; a 151936-token vocabulary goes with 3584-5120 wide
    # models), weights and hidden states random.  Shown beside it: the
    # unfused route, a cuBLAS bf16 GEMM writing the logits then the HBM-bound
    # log-prob pass (context only: library GEMM, not part of this path).
    lmh = None
    if run_lp and cid == 2 and args.lm_head_hidden > 0 and not args.no_extras:
        Hh = args.lm_head_hidden
        hid = make_hidden(4, rows, Hh, str(dev))
        wlm = make_lm_weight(4, V, Hh, str(dev))
        lws = torch.empty(tpa.lm_head_workspace_bytes(rows, V, B, T), dtype=torch.uint8, device=dev)
        lout = tuple(torch.empty_like(x) for x in lp_out)
        for _ in range(2):
            tpa.lm_head_logprobs_entropy(dtree, hid, wlm, out=lout, workspace=lws)
        reps = 3
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            tpa.lm_head_logprobs_entropy(dtree, hid, wlm, out=lout, workspace=lws)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        tpa.sync_status()
        ms_f = e0.elapsed_time(e1) / reps
        fl = 2.0 * rows * V * Hh
        torch.matmul(hid, wlm.T, out=logits)
        e0.record(stream)
        for _ in range(reps):
            torch.matmul(hid, wlm.T, out=logits)
            tpa.tree_logprobs_entropy(dtree, logits, out=lp_out)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms_u = e0.elapsed_time(e1) / reps
        lmh_peak, lmh_peak_kind = pick_bf16_peak(peaks, reps * ms_f / 1e3)
        lmh = {"rows": rows, "vocab": V, "hidden": Hh, "ms": ms_f, "tflops": fl / (ms_f / 1e3) / 1e12,
               "frac_of_bf16_peak": fl / (ms_f / 1e3) / 1e12 / lmh_peak,
               "peak": f"{peak_kind} {lmh_peak_kind} (the kernel is timed alone, {reps} launches)",
               "logits_bytes_not_written": rows * V * 2,
               "unfused_cublas_gemm_plus_logprob_ms": ms_u}
        del hid, wlm, lws, lout

    # ------------------------------------------------ end to end from host buffers
    e2e = None
    if not args.no_e2e and args.only == "all":
        pin = lambda x: x.pin_memory()
        qp, kp, vp, dop = pin(qh), pin(kh), pin(vh), pin(doh)
        lg_host = None
        if run_lp:
            lg_host = torch.empty((rows, V), dtype=torch.bfloat16, pin_memory=True)
            lg_host.copy_(logits)
        out_host = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in (o, dq, dk, dv)]
        seq_host = [torch.empty(N, dtype=torch.float32, pin_memory=True) for _ in range(2)]
        blob_buf = torch.empty(int(info.blob_bytes), dtype=torch.uint8, device=dev)

        side = torch.cuda.Stream(device=dev)
        lg_ready = torch.cuda.Event()

        # The host link moves ~210 GB/s either way whatever the stream count, so
        # the logits (15.7 GB on config 2) set the pace: they stream in on a side
        # stream while the attention inputs arrive, the attention runs and its
        # gradients go back (the other direction of the link).
        def e2e_step():
            # The copies that need no tree start first; the host packs the
            # sequences while they run.
            q.copy_(qp, non_blocking=True); k.copy_(kp, non_blocking=True)
            v.copy_(vp, non_blocking=True); do.copy_(dop, non_blocking=True)
            if run_lp:
                side.wait_stream(torch.cuda.current_stream(dev))
                with torch.cuda.stream(side):
                    logits.copy_(lg_host, non_blocking=True)
                    lg_ready.record(side)
            tr = tpa.tree_pack(tokens=toks, offsets=offs, max_tokens_per_mb=T)
            dt = tr.upload(dev, buffer=blob_buf)
            tpa.block_classify(dt, out=mask)
            tpa.tree_attn_fwd(dt, mask, q, k, v, out=o, lse=lse)
            tpa.tree_attn_bwd(dt, mask, q, k, v, o, lse, do, workspace=ws, out=(dq, dk, dv), grad_dtype=gdt)
            for h_, d_ in zip(out_host, (o, dq, dk, dv)):
                h_.copy_(d_, non_blocking=True)
            if run_lp:
                torch.cuda.current_stream(dev).wait_event(lg_ready)
                tpa.tree_logprobs_entropy(dt, logits, out=lp_out)
                seq_host[0].copy_(lp_out[2], non_blocking=True)
                seq_host[1].copy_(lp_out[3], non_blocking=True)
            torch.cuda.synchronize(dev)
            return tr

        e2e_steps = max(1, min(args.steps, args.e2e_steps))
        for _ in range(max(1, min(args.warmup, 2))):
            e2e_step()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        e2e_sec = (time.perf_counter() - t0) / e2e_steps
        if world > 1:
            tt = torch.tensor([e2e_sec], device=dev)
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
            e2e_sec = float(tt.item())
        tpa.sync_status()
        h2d = sum(x.numel() * x.element_size() for x in (qp, kp, vp, dop)) + int(info.blob_bytes) + (
            lg_host.numel() * lg_host.element_size() if lg_host is not None else 0)
        d2h = sum(x.numel() * x.element_size() for x in out_host) + (2 * 4 * N if run_lp else 0)
        e2e = {"value": job_flops / e2e_sec / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": e2e_steps, "ms_per_step": e2e_sec * 1e3,
               "includes": "pinned H2D of q,k,v,dO" + (",logits" if run_lp else "") + " (started before the host pack)"
                           " + host pack + metadata upload" +
                           " + device step + D2H of O,dQ,dK,dV" +
                           (",seq log-probs/entropies; the logits H2D overlaps the attention and its "
                            "gradients' D2H on a second stream" if run_lp else "")}

    # ------------------------------------------------ end to end with the fused LM head
    # The same attention work, but the log-prob pass starts from hidden states
    # (0.42 GB a step from pinned host memory) and the LM-head weight, resident
    # on the device like any model parameter, instead of uploading 15.7 GB of
    # logits: what a training step that owns its model would move.  Reported
    # beside `e2e` (which keeps the logits workload); it also does the LM-head
    # GEMM, which the metric does not count.
    e2e_lmh = None
    if (not args.no_e2e and args.only == "all" and run_lp and cid == 2 and args.lm_head_hidden > 0
            and not args.no_extras):
        Hh = args.lm_head_hidden
        hid_h = make_hidden(4, rows, Hh, "cpu").pin_memory()
        hid_d = torch.empty_like(hid_h, device=dev)
        wlm = make_lm_weight(4, V, Hh, str(dev))
        lws = torch.empty(tpa.lm_head_workspace_bytes(rows, V, B, T), dtype=torch.uint8, device=dev)
        pin = lambda x: x.pin_memory()
        qp, kp, vp, dop = pin(qh), pin(kh), pin(vh), pin(doh)
        out_host = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in (o, dq, dk, dv)]
        seq_host = [torch.empty(N, dtype=torch.float32, pin_memory=True) for _ in range(2)]
        blob_buf = torch.empty(int(info.blob_bytes), dtype=torch.uint8, device=dev)

        d2h = torch.cuda.Stream(device=dev)

        def e2e_lmh_step():
            # inputs that need no tree are copied while the host packs; the
            # attention results go back on a second stream during the LM head
            for d_, h_ in zip((q, k, v, do, hid_d), (qp, kp, vp, dop, hid_h)):
                d_.copy_(h_, non_blocking=True)
            tr = tpa.tree_pack(tokens=toks, offsets=offs, max_tokens_per_mb=T)
            dt = tr.upload(dev, buffer=blob_buf)
            tpa.block_classify(dt, out=mask)
            tpa.tree_attn_fwd(dt, mask, q, k, v, out=o, lse=lse)
            tpa.tree_attn_bwd(dt, mask, q, k, v, o, lse, do, workspace=ws, out=(dq, dk, dv), grad_dtype=gdt)
            d2h.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(d2h):
                for h_, d_ in zip(out_host, (o, dq, dk, dv)):
                    h_.copy_(d_, non_blocking=True)
            tpa.lm_head_logprobs_entropy(dt, hid_d, wlm, out=lp_out, workspace=lws)
            seq_host[0].copy_(lp_out[2], non_blocking=True)
            seq_host[1].copy_(lp_out[3], non_blocking=True)
            torch.cuda.synchronize(dev)
            return tr

        n_e = max(1, min(args.steps, args.e2e_steps))
        for _ in range(max(1, min(args.warmup, 2))):
            e2e_lmh_step()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(n_e):
            e2e_lmh_step()
        sec = (time.perf_counter() - t0) / n_e
        tpa.sync_status()
        h2d = sum(x.numel() * x.element_size() for x in (qp, kp, vp, dop, hid_h)) + int(info.blob_bytes)
        d2h = sum(x.numel() * x.element_size() for x in out_host) + 2 * 4 * N
        e2e_lmh = {"value": job_flops / sec / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
                   "d2h_bytes_per_step": d2h, "steps": n_e, "ms_per_step": sec * 1e3, "hidden": Hh,
                   "includes": "pinned H2D of q,k,v,dO and hidden states (overlapping the host pack) + metadata "
                               "upload + device step with the fused LM-head log-prob pass (weight resident) + D2H of "
                               "O,dQ,dK,dV (on a second stream, overlapping the LM head), seq log-probs/entropies"}
        del hid_h, hid_d, wlm, lws

    timed_s = total_ms / 1e3
    bf16_peak, bf16_kind = pick_bf16_peak(peaks, timed_s)
    rate = lambda work, ms: work / (ms / 1e3) if ms > 1e-6 else 0.0
    attn_tflops = rate(flops_step / 1e12, t_fwd + t_bwd)
    bwd_tflops = rate(flops_bwd / 1e12, t_bwd)
    fwd_tflops = rate(flops_fwd / 1e12, t_fwd)
    lp_bytes = rows * V * 2 + 4 * 4 * B * T + 8 * N
    lp_gbs = rate(lp_bytes / 1e9, t_lp)
    kernel_ms = {"tpa_tree_attn_bwd": t_bwd if run_attn else 0.0, "tpa_tree_attn_fwd": t_fwd if run_attn else 0.0,
                 "tpa_tree_logprobs_entropy": t_lp if run_lp else 0.0}
    dominant = max(kernel_ms.items(), key=lambda x: x[1])[0]

    def tensor_roof(entry, achieved, work):
        return {"bound": "tensor", "achieved": achieved, "peak": bf16_peak, "unit": "TFLOP/s",
                "frac": achieved / bf16_peak, "traffic": _profile_traffic(entry, rows),
                "traffic_unit": "bytes per launch (ncu DRAM read + write, scaled by tree tokens)",
                "kernel": entry, "peak_kind": f"{peak_kind} {bf16_kind} (timed region {timed_s:.2f} s)",
                "algorithmic_per_launch": work}

    lp_roof = None
    if run_lp:
        lp_roof = {"bound": "hbm", "achieved": lp_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                   "frac": lp_gbs / peaks["hbm_gbs"], "frac_of_nominal_8tbs": lp_gbs / NOMINAL_HBM_GBS,
                   "traffic": _profile_traffic("tpa_tree_logprobs_entropy", rows),
                   "traffic_unit": "bytes per launch (ncu DRAM read + write, scaled by tree tokens)",
                   "kernel": "tpa_tree_logprobs_entropy", "peak_kind": f"{peak_kind} HBM copy",
                   "algorithmic_per_launch": lp_bytes}
    if dominant == "tpa_tree_logprobs_entropy":
        roof = lp_roof
    elif dominant == "tpa_tree_attn_bwd":
        roof = tensor_roof(dominant, bwd_tflops, flops_bwd)
    else:
        roof = tensor_roof(dominant, fwd_tflops, flops_fwd)

    # Micro-batch / rank balancing (host): the blog post's experiment shape —
    # the workload's sequences split over 4 ranks with unbounded capacity —
    # FFD against KK spread, and the cost of one call.
    bal = None
    if rank == 0 and not args.no_extras:
        lens = [len(s_) for s_ in seqs]
        bal = {"items": len(lens), "groups": 4}
        for algo in ("ffd", "kk"):
            t0 = time.perf_counter()
            for _ in range(20):
                g_, ng_, used_ = tpa.balance(lens, 10**12, 4, 1, algo)
            bal[f"{algo}_us_per_call"] = (time.perf_counter() - t0) / 20 * 1e6
            bal[f"{algo}_spread"] = tpa.packing_metrics(lens, g_, ng_, 10**12)["spread"]
        bal["kk_improvement_pct"] = (100.0 * (bal["ffd_spread"] - bal["kk_spread"]) / bal["ffd_spread"]
                                     if bal["ffd_spread"] else 0.0)
        # host steps 1-3 of tree building on the workload as a right-padded batch
        L = max(lens)
        ids = np.zeros((len(seqs), L), dtype=np.int32)
        am = np.zeros((len(seqs), L), dtype=np.uint8)
        for r_, s_ in enumerate(seqs):
            ids[r_, :len(s_)] = s_
            am[r_, :len(s_)] = 1
        t0 = time.perf_counter()
        for _ in range(5):
            tpa.extract_sequences(ids, am)
        t1 = time.perf_counter()
        for _ in range(5):
            tpa.tree_pack(tokens=toks, offsets=offs, max_tokens_per_mb=T)
        t2 = time.perf_counter()
        for _ in range(5):
            tpa.tree_pack_padded(ids, am, T)
        t3 = time.perf_counter()
        bal["host_ms"] = {"extract": (t1 - t0) / 5 * 1e3, "pack": (t2 - t1) / 5 * 1e3,
                          "pack_padded": (t3 - t2) / 5 * 1e3, "padded_batch": list(ids.shape)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.only == "all":
        r = cpu_oracle_run(1, 0, args.oracle_pairs, cid)
        side = cpu_oracle_side(cid, V if run_lp else None)
        cpu = {"value": r["value"], "unit": UNIT, "cores": r["cores"], "kind": "oracle", "sample": r["sample"],
               "tree_tokens_per_s": r["tree_tokens_per_s"], **side}

    value = job_flops / (ms_step / 1e3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOADS[cid], "config_id": cid, "n_trees": B, "tree_tokens": rows,
                   "original_tokens": int(N), "tree_token_ratio": info.tree_token_ratio, "ancestor_pairs": pairs,
                   "flops_per_step": flops_step, "flops_per_step_strict_12PdHq": flops_strict,
                   "grad_dtype": args.grad_dtype,
                   "l2": ("inputs larger than L2 (129 MB); no flush" if flush is None else
                          "256 MB buffer written between steps to flush the L2 (outside the timed segments)"),
                   "parallelism": (f"trees split over {world} ranks by KK balancing of ancestor pairs"
                                   if world > 1 else "single GPU")},
        "tree_tokens_per_s": job_rows / (ms_step / 1e3),
        "original_token_equiv_per_s": N * (job_rows / max(rows, 1)) / (ms_step / 1e3),
        "frac_of_bf16_peak": value / bf16_peak,
        "breakdown_ms": {"block_classify": t_cls, "attn_fwd": t_fwd, "attn_bwd": t_bwd, "logprobs_entropy": t_lp,
                         "stat": "median over the timed steps"},
        "breakdown_spread_ms": stats,
        "attn_fwd_bwd_tflops": attn_tflops, "attn_fwd_bwd_tflops_strict": rate(flops_strict / 1e12, t_fwd + t_bwd),
        "attn_fwd_tflops": fwd_tflops, "attn_bwd_tflops": bwd_tflops,
        "attn_fwd_bwd_frac_of_bf16_peak": attn_tflops / bf16_peak, "bf16_peak_used": bf16_kind,
        "logprobs_gbs": lp_gbs if run_lp else None,
        "logprobs_frac_hbm": lp_gbs / peaks["hbm_gbs"] if run_lp else None,
        "logprobs_frac_nominal_8tbs": lp_gbs / NOMINAL_HBM_GBS if run_lp else None,
        "roofline": roof, "roofline_logprobs": lp_roof, "clocks": clocks,
        "attn_gcycles_at_median_clock": ((t_fwd + t_bwd) * clocks["sm_mhz"] / 1e6) if clocks["sm_mhz"] else None,
        "gpu_launches": n_launch_per_step * args.steps,
        "e2e": e2e, "e2e_lm_head": e2e_lmh, "cpu_baseline": cpu, "balance": bal, "lm_head": lmh,
        "dense_mask": None if dmask is None else {
            **dmask, "frac_hbm_u8": dmask["u8"]["gbs"] / peaks["hbm_gbs"],
            "note": "write-only export of the [B, T, T] ancestor mask (u8) and its bit-packed form; "
                    "fraction against the measured copy bandwidth"},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, choices=[1, 2, 3, 5], default=2,
                    help="workload: 1 tiny, 2 GRPO-shaped with the log-prob pass (headline), 3 agentic, "
                         "5 large few-shot")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--lm-head-hidden", type=int, default=4096,
                    help="hidden size of the fused LM-head measurement (0 skips it)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the measurements outside the step (dense mask, LM head, balancing)")
    ap.add_argument("--grad-dtype", choices=["bf16", "fp32"], default="bf16",
                    help="dtype of dQ, dK, dV (bf16 as the workload's tensors; fp32 for the split-column path)")
    ap.add_argument("--oracle-pairs", type=int, default=15000000,
                    help="ancestor pairs in the oracle's bounded sample")
    ap.add_argument("--only", choices=["all", "attn", "logprobs"], default="all",
                    help="profiling aid: run only part of the step (no e2e / CPU baseline then)")
    ap.add_argument("--max-trees", type=int, default=0,
                    help="profiling aid: keep only the sequences of the first N trees")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    rank, world, local = _dist()
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" and torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_gpu(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
