"""Oracle fp64 log-probabilities and entropies (test infrastructure).

From the AReaL "树训练" page, §对数概率计算 (log-probability computation): in a
packed tree the labels cannot be obtained by rolling ``input_ids`` (sequences
share positions); each sequence must recover its own token order from the
tree, and the per-node results (within-node predictions and the transition
to a child node) are only a cache. The plain definition, computed here
sequence by sequence with no caching:

    for sequence s = (x_0 .. x_{L-1}) placed at tree positions g_0 .. g_{L-1}:
        ls_t      = log_softmax(logits[row(g_t)])            (fp64)
        logp_s[t] = ls_t[x_{t+1}]   for t < L - 1,   0 at t = L - 1
        ent_s[t]  = - sum_v exp(ls_t[v]) ls_t[v]

Readings: the last position of each sequence has no label and gets 0 (the
rolled-label convention); entropy uses the natural log, and a vocabulary
entry with p = 0 (a logit of -inf, e.g. a masked token) contributes 0 to it,
the limit of p log p as p -> 0. ``row(g)`` is the logits row of tree
position g: ``row_base[tree] + g``.
"""
from __future__ import annotations

import numpy as np
import torch

from .pack import OraclePacking


def _log_softmax64(rows: torch.Tensor) -> torch.Tensor:
    x = rows.to(torch.float64)
    m = x.max(dim=-1, keepdim=True).values
    z = x - m
    return z - torch.log(torch.exp(z).sum(dim=-1, keepdim=True))


def _entropy64(ls: torch.Tensor) -> torch.Tensor:
    """-sum_v p_v log p_v over the last axis from log-probabilities ``ls``;
    entries with p = 0 (ls = -inf) are left out of the sum (0 log 0 = 0)."""
    plogp = torch.exp(ls) * ls
    return -torch.where(torch.isneginf(ls), torch.zeros_like(plogp), plogp).sum(-1)


def sequence_logprobs_entropy(pk: OraclePacking, seqs: list[list[int]], logits: torch.Tensor,
                              row_base: list[int], seq_ids: list[int] | None = None):
    """Per-sequence fp64 log-probs and entropies.

    ``logits`` is indexable by row (a CPU tensor ``[rows, V]``); returns two
    lists of fp64 numpy arrays, one entry per requested sequence."""
    ids = range(len(seqs)) if seq_ids is None else seq_ids
    out_lp, out_ent = [], []
    for s in ids:
        b = int(pk.seq_tree[s])
        rows = torch.as_tensor(row_base[b] + pk.seq_pos[s], dtype=torch.long)
        ls = _log_softmax64(logits[rows])
        L = len(seqs[s])
        lp = np.zeros(L, dtype=np.float64)
        if L > 1:
            nxt = torch.as_tensor(seqs[s][1:], dtype=torch.long)
            lp[:-1] = ls[torch.arange(L - 1), nxt].numpy()
        ent = _entropy64(ls).numpy()
        out_lp.append(lp)
        out_ent.append(ent)
    return out_lp, out_ent


def position_logprobs_entropy(pk: OraclePacking, logits: torch.Tensor, row_base: list[int],
                              tree: int, positions: list[int] | None = None):
    """Node-level values at tree positions: for each position p, the entropy
    of row(p) and the log-prob of the token at p under its parent's row
    (0 where p has no parent). This is the cache the page describes, written
    out per position."""
    t = pk.trees[tree]
    pos = range(t.n) if positions is None else positions
    ent = np.zeros(len(pos))
    lp = np.zeros(len(pos))
    for u, p in enumerate(pos):
        ls = _log_softmax64(logits[row_base[tree] + p][None])[0]
        ent[u] = float(_entropy64(ls))
        par = int(t.parent[p])
        if par >= 0:
            lsp = _log_softmax64(logits[row_base[tree] + par][None])[0]
            lp[u] = float(lsp[int(t.tokens[p])])
    return lp, ent
