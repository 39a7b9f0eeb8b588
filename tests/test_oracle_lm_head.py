"""Pins for the oracle LM-head logits (logits[r, v] = sum_k h[r, k] w[v, k])
feeding the pinned §对数概率计算 log-prob oracle."""
import math

import numpy as np
import torch

import oracle
from oracle.lm_head import LazyLogits
from oracle.logprobs import sequence_logprobs_entropy


def test_hand_example_orientation():
    h = torch.tensor([[1.0, 0.0], [0.0, 2.0]])
    w = torch.tensor([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])
    lg = LazyLogits(h, w)[torch.tensor([0, 1])]
    assert lg.tolist() == [[1.0, 0.0, 1.0], [0.0, 2.0, 2.0]]


def test_matches_explicit_sum():
    g = torch.Generator().manual_seed(0)
    h = torch.randn(5, 7, generator=g).to(torch.bfloat16)
    w = torch.randn(11, 7, generator=g).to(torch.bfloat16)
    lg = LazyLogits(h, w)[torch.arange(5)]
    for r in range(5):
        for v in range(11):
            s = sum(float(h[r, k]) * float(w[v, k]) for k in range(7))
            assert abs(float(lg[r, v]) - s) < 1e-12


def test_zero_weight_gives_uniform_distribution():
    seqs = [[0, 1, 2], [0, 1, 3]]
    pk = oracle.tree_pack(seqs, 128)
    V = 9
    lg = LazyLogits(torch.randn(pk.total_tree_tokens, 4), torch.zeros(V, 4))
    lp, ent = sequence_logprobs_entropy(pk, seqs, lg, [0])
    for s in range(2):
        assert np.allclose(ent[s], math.log(V))
        assert np.allclose(lp[s][:-1], -math.log(V)) and lp[s][-1] == 0.0
