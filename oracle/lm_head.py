"""Oracle LM-head log-probabilities (test infrastructure; see the package
docstring).

The step upstream of the tree training page's §对数概率计算: the logits of a
tree row are the LM head applied to that row's hidden state,

    logits[r, v] = sum_k hidden[r, k] * weight[v, k]      (fp64),

with ``hidden`` [rows, H] and ``weight`` [V, H] the exact bf16 values widened
to fp64; log-probs and entropies then follow the §对数概率计算 definition of
``logprobs`` unchanged.  ``LazyLogits`` computes only the rows a check asks
for, so full-vocabulary rows can be sampled at any size.
"""
from __future__ import annotations

import torch


class LazyLogits:
    """Row-indexable fp64 logits ``hidden @ weight.T`` computed on demand."""

    def __init__(self, hidden: torch.Tensor, weight: torch.Tensor):
        self.hidden = hidden
        self.weight64 = weight.to(torch.float64)

    def __getitem__(self, rows):
        h = self.hidden[rows].to(torch.float64)
        return h @ self.weight64.T
