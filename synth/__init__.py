"""Seeded synthetic workloads for prefix-shared tree attention.

This module holds ONLY random input generators: token sequences with the
sharing structure of RL rollouts, and the q/k/v/dO/logits tensors that go
with them. It contains none of the method's arithmetic (no trie, no mask,
no attention, no log-softmax), so both the CUDA path's tests and the CPU
oracle's tests may draw their inputs from it.

Workload shapes follow the tree-training page (AReaL "树训练": the worked
example in "树构建过程" and the RL settings listed in "概述": several samples
per prompt, shared system prompts or few-shot examples, multi-turn history)
and the micro-batch packing blog post (its bimodal length generator,
"何时使用 KK": short 50-200 and long 800-2048 tokens, 30 % long).

Structure randomness uses ``numpy.random.default_rng(seed)``; tensors use a
CPU ``torch.Generator`` seeded ``1000 * config + t`` (t = 1 q, 2 k, 3 v,
4 dO, 5 logits) so that every consumer sees identical values.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "WorkloadConfig",
    "CONFIGS",
    "make_sequences",
    "make_qkv",
    "make_dout",
    "make_logits",
    "random_small_sequences",
    "flatten_sequences",
]


@dataclass(frozen=True)
class WorkloadConfig:
    """Sizes of one synthetic workload."""

    cid: int
    name: str
    max_tokens_per_mb: int
    n_heads_q: int
    n_heads_kv: int
    head_dim: int
    vocab: int            # token-id range of the sequences
    logits_vocab: int     # vocabulary width of the logits tensor
    extra: dict = field(default_factory=dict)


CONFIGS: dict[int, WorkloadConfig] = {
    1: WorkloadConfig(1, "tiny: 4 prompts x 4 samples, vocab 1000, mb 1024, 4/4 heads, d 64",
                      1024, 4, 4, 64, 1000, 1000),
    2: WorkloadConfig(2, "GRPO-shaped: 8 prompts x 8 samples, bimodal responses, mb 8192, 32/8 heads, d 128",
                      8192, 32, 8, 128, 32000, 151936),
    3: WorkloadConfig(3, "agentic multi-turn: 2048-token system prompt, 16 branching trajectories, mb 32768, 16/2 heads, d 128",
                      32768, 16, 2, 128, 32000, 151936),
    4: WorkloadConfig(4, "log-prob/entropy gather: config-2 trees, logits width 151936",
                      8192, 32, 8, 128, 32000, 151936),
    5: WorkloadConfig(5, "large few-shot tree: 4096-token shared prefix, 64 samples, mb 65536, 32/8 heads, d 128",
                      65536, 32, 8, 128, 32000, 151936),
}


def _ids(rng: np.random.Generator, n: int, vocab: int) -> list[int]:
    return rng.integers(0, vocab, size=n).tolist()


def _config1(rng: np.random.Generator) -> list[list[int]]:
    seqs = []
    for _ in range(4):
        prompt = _ids(rng, 64, 1000)
        for _ in range(4):
            n = int(rng.integers(16, 65))
            seqs.append(prompt + _ids(rng, n, 1000))
    return seqs


def _config2(rng: np.random.Generator) -> list[list[int]]:
    seqs = []
    for _ in range(8):
        prompt = _ids(rng, int(rng.integers(256, 1025)), 32000)
        for _ in range(8):
            if rng.random() < 0.3:
                n = int(rng.integers(800, 2049))
            else:
                n = int(rng.integers(50, 201))
            seqs.append(prompt + _ids(rng, n, 32000))
    return seqs


def _config3(rng: np.random.Generator) -> list[list[int]]:
    system = _ids(rng, 2048, 32000)
    turns: list[list[int]] = []          # turn id -> tokens
    trajs: list[list[int]] = []          # trajectory -> list of turn ids
    children: dict[tuple, set] = {}      # branch point (tuple of turn ids) -> next turn ids

    def fresh_turn() -> int:
        turns.append(_ids(rng, int(rng.integers(64, 513)), 32000))
        return len(turns) - 1

    for i in range(16):
        n_i = int(rng.integers(4, 9))
        if i == 0:
            shared: list[int] = []
        else:
            shared = []
            for _attempt in range(1000):
                j = int(rng.integers(0, i))
                b = int(rng.integers(0, min(n_i, len(trajs[j]))))
                key = tuple(trajs[j][:b])
                if len(children.get(key, ())) < 3:
                    shared = trajs[j][:b]
                    break
            else:  # every draw hit a full branch point: share nothing extra
                shared = []
        traj = list(shared)
        while len(traj) < n_i:
            traj.append(fresh_turn())
        for b in range(len(traj)):
            children.setdefault(tuple(traj[:b]), set()).add(traj[b])
        trajs.append(traj)
    seqs = []
    for traj in trajs:
        s = list(system)
        for t in traj:
            s.extend(turns[t])
        seqs.append(s)
    return seqs


def _config5(rng: np.random.Generator) -> list[list[int]]:
    prefix = _ids(rng, 4096, 32000)
    depths = np.sort(rng.choice(4096, size=16, replace=False))
    conts: list[list[int]] = []
    for i in range(64):
        L = int(rng.integers(512, 4097))
        if i == 0:
            conts.append(_ids(rng, L, 32000))
            continue
        j = int(rng.integers(0, i))
        lim = min(L, len(conts[j]))
        below = depths[depths < lim]
        d = int(below[-1]) if below.size else 0
        conts.append(conts[j][:d] + _ids(rng, L - d, 32000))
    return [prefix + c for c in conts]


_BUILDERS = {1: _config1, 2: _config2, 3: _config3, 4: _config2, 5: _config5}


def make_sequences(cid: int, seed: int | None = None) -> list[list[int]]:
    """Token sequences of workload ``cid`` (config 4 reuses config 2's
    generator); ``seed`` defaults to the config id (config 4: seed 2)."""
    if seed is None:
        seed = 2 if cid == 4 else cid
    return _BUILDERS[cid](np.random.default_rng(seed))


def flatten_sequences(seqs: list[list[int]]) -> tuple[np.ndarray, np.ndarray]:
    """Concatenated int32 tokens and int64 offsets ``[n + 1]``."""
    offs = np.zeros(len(seqs) + 1, dtype=np.int64)
    offs[1:] = np.cumsum([len(s) for s in seqs])
    toks = np.fromiter((t for s in seqs for t in s), dtype=np.int32, count=int(offs[-1]))
    return toks, offs


def random_small_sequences(rng: np.random.Generator, n_seqs: int, max_len: int,
                           vocab: int, min_len: int = 1) -> list[list[int]]:
    """Tiny random sequences over a small vocabulary, which forces heavy
    prefix sharing (used for brute-force checks)."""
    return [rng.integers(0, vocab, size=int(rng.integers(min_len, max_len + 1))).tolist()
            for _ in range(n_seqs)]


def _gen(cid: int, t: int):
    import torch
    g = torch.Generator(device="cpu")
    g.manual_seed(1000 * cid + t)
    return g


def make_qkv(cid: int, n_trees: int, t_pad: int, hq: int, hkv: int, d: int):
    """q ``[B, T_pad, Hq, d]``, k and v ``[B, T_pad, Hkv, d]``, bf16, N(0, 1)
    (pad positions hold finite random values too)."""
    import torch
    q = torch.randn((n_trees, t_pad, hq, d), generator=_gen(cid, 1)).to(torch.bfloat16)
    k = torch.randn((n_trees, t_pad, hkv, d), generator=_gen(cid, 2)).to(torch.bfloat16)
    v = torch.randn((n_trees, t_pad, hkv, d), generator=_gen(cid, 3)).to(torch.bfloat16)
    return q, k, v


def make_dout(cid: int, n_trees: int, t_pad: int, hq: int, d: int):
    """Upstream gradient dO ``[B, T_pad, Hq, d]`` bf16, N(0, 1)."""
    import torch
    return torch.randn((n_trees, t_pad, hq, d), generator=_gen(cid, 4)).to(torch.bfloat16)


def make_logits(cid: int, rows: int, vocab: int, device: str = "cpu", chunk_rows: int = 4096):
    """Logits ``[rows, vocab]`` bf16 drawn from N(0, 2^2), i.e. ``2 * randn``.

    On CPU the values come from ``torch.Generator`` seeded ``1000 * cid + 5``.
    On a CUDA device a CUDA generator with the same seed is used (values differ
    from the CPU draw; consumers copy the rows they need back to the host)."""
    import torch
    out = torch.empty((rows, vocab), dtype=torch.bfloat16, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(1000 * cid + 5)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        out[r0:r1] = (2.0 * torch.randn((r1 - r0, vocab), generator=g, device=device)).to(torch.bfloat16)
    return out


def make_hidden(cid: int, rows: int, hidden: int, device: str = "cpu"):
    """Hidden states ``[rows, hidden]`` bf16 ~ N(0, 1) (the LM head's input),
    from a ``torch.Generator`` on ``device`` seeded ``1000 * cid + 6``."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(1000 * cid + 6)
    return torch.randn((rows, hidden), generator=g, device=device).to(torch.bfloat16)


def make_lm_weight(cid: int, vocab: int, hidden: int, device: str = "cpu"):
    """LM-head weight ``[vocab, hidden]`` bf16 ~ N(0, (2 / sqrt(hidden))^2), so
    that logits of N(0, 1) hidden states have standard deviation 2 like the
    logits workload; ``torch.Generator`` on ``device`` seeded ``1000 * cid + 7``."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(1000 * cid + 7)
    return (torch.randn((vocab, hidden), generator=g, device=device) * (2.0 / hidden ** 0.5)).to(torch.bfloat16)
