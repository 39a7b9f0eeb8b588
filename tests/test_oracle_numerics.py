"""Pins for the oracle mask, block classes, attention and log-probs (CPU).

Attention is pinned by the page's own invariant (a token sees exactly its
ancestors, so each sequence's rows equal plain causal attention over that
sequence alone) checked against torch's fp64 causal
``scaled_dot_product_attention`` and its autograd; block classes by
closed-form cases; log-probs by closed forms and by ``cross_entropy``.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle.mask import (EMPTY, FULL, PARTIAL, _mask_rows, ancestor_pairs, block_classes,
                         block_classes_dense, block_csr, dense_mask)
from synth import random_small_sequences


def _gqa_causal(q, k, v, scale):
    """Causal attention of one sequence via torch SDPA in fp64: q [L,Hq,d],
    k/v [L,Hkv,d].  The query-head to key/value-head mapping is torch's own
    grouped-query attention (``enable_gqa``), not a repeat written here."""
    return F.scaled_dot_product_attention(q.transpose(0, 1)[None], k.transpose(0, 1)[None],
                                          v.transpose(0, 1)[None], is_causal=True, scale=scale,
                                          enable_gqa=True)[0].transpose(0, 1)


def _bf16_randn(shape, g):
    return torch.randn(shape, generator=g).to(torch.bfloat16).to(torch.float64)


# ---------------------------------------------------------------- mask / blocks

@pytest.mark.parametrize("seed", range(10))
def test_interval_rows_equal_parent_walk(seed):
    rng = np.random.default_rng(seed)
    seqs = random_small_sequences(rng, 10, 40, 3)
    t = oracle.tree_pack(seqs, 512).trees[0]
    M = dense_mask(t, 512)
    assert np.array_equal(_mask_rows(t, 0, 512, 512), M)
    assert np.array_equal(block_classes(t, 512), block_classes_dense(M))
    assert ancestor_pairs(t) == int(M.sum())


def test_block_classes_closed_form_chain():
    # one sequence of 300 tokens in T_pad = 384: causal lower triangle
    t = oracle.tree_pack([list(range(300))], 384).trees[0]
    cls = block_classes(t, 384)
    expect = np.array([[PARTIAL, EMPTY, EMPTY],
                       [FULL, PARTIAL, EMPTY],
                       [PARTIAL, PARTIAL, PARTIAL]], dtype=np.uint8)   # 44 real queries in block 2
    assert np.array_equal(cls, expect)
    csr = block_csr(cls)
    assert csr["q_ptr"].tolist() == [0, 1, 3, 6]
    assert csr["q_idx"].tolist() == [0, 1, 2, 0, 2, 4]
    assert csr["k_ptr"].tolist() == [0, 3, 5, 6]
    assert csr["k_idx"].tolist() == [0, 3, 4, 2, 4, 4]


def test_block_classes_two_branches():
    # shared 128-token prefix then two 128-token branches: block (2,1) is empty
    pre = list(range(128))
    a = pre + [1000 + i for i in range(128)]
    b = pre + [2000 + i for i in range(128)]
    t = oracle.tree_pack([a, b], 512).trees[0]
    cls = block_classes(t, 512)
    assert cls[1, 0] == FULL and cls[2, 0] == FULL
    assert cls[2, 1] == EMPTY and cls[1, 1] == PARTIAL and cls[2, 2] == PARTIAL
    assert np.all(cls[3] == EMPTY)


# ---------------------------------------------------------------- attention

def _random_case(seed, hq, hkv, d, max_len=24, vocab=3, n=6, mb=128):
    rng = np.random.default_rng(seed)
    seqs = random_small_sequences(rng, n, max_len, vocab)
    pk = oracle.tree_pack(seqs, mb)
    g = torch.Generator().manual_seed(seed)
    B, T = pk.n_trees, mb
    q = _bf16_randn((B, T, hq, d), g)
    k = _bf16_randn((B, T, hkv, d), g)
    v = _bf16_randn((B, T, hkv, d), g)
    dO = _bf16_randn((B, T, hq, d), g)
    return seqs, pk, q, k, v, dO


def test_chain_equals_sdpa_causal():
    g = torch.Generator().manual_seed(0)
    L, T = 150, 256
    t = oracle.tree_pack([list(range(L))], T).trees[0]
    q = _bf16_randn((T, 4, 64), g)
    k = _bf16_randn((T, 2, 64), g)
    v = _bf16_randn((T, 2, 64), g)
    O, LSE = oracle.attn_forward(t, q, k, v, t_pad=T)
    ref = _gqa_causal(q[:L], k[:L], v[:L], 1 / 8)
    assert torch.allclose(O[:L], ref, atol=1e-12, rtol=1e-12)
    assert torch.all(O[L:] == 0) and torch.all(LSE[:, L:] == 0)
    S = torch.einsum("ihd,jhd->hij", q[:L], k[:L].repeat_interleave(2, 1)) / 8
    S = S.masked_fill(~torch.tril(torch.ones(L, L, dtype=torch.bool)), float("-inf"))
    assert torch.allclose(LSE[:, :L], torch.logsumexp(S, -1), atol=1e-12)


@pytest.mark.parametrize("seed,hq,hkv,d", [(1, 2, 2, 16), (2, 4, 2, 16), (3, 4, 1, 32), (4, 6, 3, 8)])
def test_per_sequence_invariant_forward(seed, hq, hkv, d):
    seqs, pk, q, k, v, _ = _random_case(seed, hq, hkv, d)
    outs = [oracle.attn_forward(t, q[b], k[b], v[b], t_pad=128) for b, t in enumerate(pk.trees)]
    for s, seq in enumerate(seqs):
        b = int(pk.seq_tree[s])
        pos = torch.from_numpy(pk.seq_pos[s])
        ref = _gqa_causal(q[b][pos], k[b][pos], v[b][pos], 1 / math.sqrt(d))
        assert torch.allclose(outs[b][0][pos], ref, atol=1e-12, rtol=1e-10)


@pytest.mark.parametrize("seed,hq,hkv,d", [(5, 2, 2, 16), (6, 4, 2, 16), (7, 4, 1, 8)])
def test_per_sequence_invariant_backward(seed, hq, hkv, d):
    # Tree gradients with tree dO = scatter-sum of per-sequence dO must equal
    # the scatter-sum of per-sequence causal-attention gradients.
    seqs, pk, q, k, v, _ = _random_case(seed, hq, hkv, d)
    g = torch.Generator().manual_seed(seed + 1000)
    B, T = pk.n_trees, 128
    dq_ref = torch.zeros_like(q)
    dk_ref = torch.zeros_like(k)
    dv_ref = torch.zeros_like(v)
    dO_tree = torch.zeros_like(q)
    for s, seq in enumerate(seqs):
        b = int(pk.seq_tree[s])
        pos = torch.from_numpy(pk.seq_pos[s])
        qs = q[b][pos].clone().requires_grad_(True)
        ks = k[b][pos].clone().requires_grad_(True)
        vs = v[b][pos].clone().requires_grad_(True)
        out = _gqa_causal(qs, ks, vs, 1 / math.sqrt(d))
        dos = _bf16_randn(out.shape, g)
        out.backward(dos)
        dq_ref[b].index_add_(0, pos, qs.grad)
        dk_ref[b].index_add_(0, pos, ks.grad)
        dv_ref[b].index_add_(0, pos, vs.grad)
        dO_tree[b].index_add_(0, pos, dos)
    for b, t in enumerate(pk.trees):
        dq, dk, dv = oracle.attn_backward(t, q[b], k[b], v[b], dO_tree[b], t_pad=T)
        assert torch.allclose(dq, dq_ref[b], atol=1e-10)
        assert torch.allclose(dk, dk_ref[b], atol=1e-10)
        assert torch.allclose(dv, dv_ref[b], atol=1e-10)


@pytest.mark.parametrize("hq,hkv", [(4, 2), (6, 3), (8, 1), (6, 2)])
def test_gqa_head_mapping_by_hand(hq, hkv):
    # Query head h reads key/value head h // (hq // hkv): each head of a
    # single-sequence tree is compared with a one-head causal attention whose
    # key/value head is picked by that formula, one head at a time.
    g = torch.Generator().manual_seed(40 + hq + hkv)
    L, d = 70, 16
    t = oracle.tree_pack([list(range(L))], 128).trees[0]
    q = _bf16_randn((128, hq, d), g)
    k = _bf16_randn((128, hkv, d), g)
    v = _bf16_randn((128, hkv, d), g)
    O, _ = oracle.attn_forward(t, q, k, v, t_pad=128)
    group = hq // hkv
    for h in range(hq):
        kv = h // group
        S = (q[:L, h] @ k[:L, kv].T) / math.sqrt(d)
        S = S.masked_fill(~torch.tril(torch.ones(L, L, dtype=torch.bool)), float("-inf"))
        ref = torch.softmax(S, -1) @ v[:L, kv]
        assert torch.allclose(O[:L, h], ref, atol=1e-12), f"head {h}"
        # and no other key/value head gives it (the heads' values differ)
        for other in range(hkv):
            if other != kv:
                alt = torch.softmax(((q[:L, h] @ k[:L, other].T) / math.sqrt(d)).masked_fill(
                    ~torch.tril(torch.ones(L, L, dtype=torch.bool)), float("-inf")), -1) @ v[:L, other]
                assert not torch.allclose(O[:L, h], alt, atol=1e-6)


def test_node_subset_matches_full():
    seqs, pk, q, k, v, dO = _random_case(11, 4, 2, 16, n=8)
    t = pk.trees[0]
    O, L = oracle.attn_forward(t, q[0], k[0], v[0], t_pad=128)
    nodes = [0, len(t.node_start) - 1]
    Os, Ls = oracle.attn_forward(t, q[0], k[0], v[0], t_pad=128, nodes=nodes)
    for nid in nodes:
        s0, s1 = t.node_start[nid], t.node_end[nid] + 1
        assert torch.equal(Os[s0:s1], O[s0:s1]) and torch.equal(Ls[:, s0:s1], L[:, s0:s1])


# ---------------------------------------------------------------- log-probs

def test_logprobs_closed_form_uniform():
    seqs = [[0, 1, 2], [0, 1, 3]]
    pk = oracle.tree_pack(seqs, 128)
    V = 7
    logits = torch.full((pk.trees[0].n, V), 0.25)
    lp, ent = oracle.sequence_logprobs_entropy(pk, seqs, logits, [0])
    for s in range(2):
        assert np.allclose(lp[s][:-1], -math.log(V)) and lp[s][-1] == 0.0
        assert np.allclose(ent[s], math.log(V))


def test_logprobs_closed_form_spike():
    seqs = [[2, 5, 1]]
    pk = oracle.tree_pack(seqs, 128)
    V, a = 6, 3.0
    logits = torch.zeros((3, V), dtype=torch.float64)
    logits[:, 1] = a                      # token 1 is favoured at every row
    lp, ent = oracle.sequence_logprobs_entropy(pk, seqs, logits, [0])
    Z = math.exp(a) + V - 1
    assert lp[0][0] == pytest.approx(-math.log(Z))          # label 5 (not the spike)
    assert lp[0][1] == pytest.approx(a - math.log(Z))       # label 1 (the spike)
    p1 = math.exp(a) / Z
    H = -p1 * math.log(p1) - (V - 1) / Z * math.log(1 / Z)
    assert np.allclose(ent[0], H)


@pytest.mark.parametrize("seed", range(4))
def test_logprobs_vs_cross_entropy_and_cache(seed):
    rng = np.random.default_rng(seed)
    seqs = random_small_sequences(rng, 7, 15, 3, min_len=2)
    pk = oracle.tree_pack(seqs, 128)
    V = 11
    rows = sum(t.n for t in pk.trees)
    row_base = np.concatenate([[0], np.cumsum([t.n for t in pk.trees])])[:-1].tolist()
    logits = 2 * torch.randn((rows, V), generator=torch.Generator().manual_seed(seed), dtype=torch.float64)
    lp, ent = oracle.sequence_logprobs_entropy(pk, seqs, logits, row_base)
    for s, seq in enumerate(seqs):
        b = int(pk.seq_tree[s])
        r = torch.as_tensor(row_base[b] + pk.seq_pos[s])
        ce = F.cross_entropy(logits[r[:-1]], torch.as_tensor(seq[1:]), reduction="none")
        assert np.allclose(lp[s][:-1], -ce.numpy(), atol=1e-12)
        p = torch.softmax(logits[r], -1)
        assert np.allclose(ent[s], (-(p * torch.log(p)).sum(-1)).numpy(), atol=1e-12)
        # node-level values gathered along the sequence give the same numbers
        plp, pent = oracle.position_logprobs_entropy(pk, logits, row_base, b, pk.seq_pos[s].tolist())
        assert np.allclose(pent, ent[s], atol=1e-12)
        assert np.allclose(plp[1:], lp[s][:-1], atol=1e-12)


def test_logprobs_masked_entries_closed_form():
    # k equal finite logits and the rest -inf: a uniform distribution over k
    # entries, entropy log k; a label at a finite entry has log-prob -log k,
    # a label at a masked entry -inf.
    seqs = [[0, 3, 5, 3]]
    pk = oracle.tree_pack(seqs, 128)
    V = 9
    logits = torch.full((4, V), float("-inf"), dtype=torch.float64)
    logits[:, [1, 3, 4, 7]] = 0.5                   # k = 4 finite entries, token 5 masked
    lp, ent = oracle.sequence_logprobs_entropy(pk, seqs, logits, [0])
    assert np.allclose(ent[0], math.log(4))
    assert lp[0][0] == pytest.approx(-math.log(4))    # label 3
    assert lp[0][1] == float("-inf")                   # label 5 is masked
    assert lp[0][2] == pytest.approx(-math.log(4)) and lp[0][3] == 0.0


@pytest.mark.parametrize("seed", range(3))
def test_logprobs_masked_entries_vs_scipy_entr(seed):
    # Random rows with scattered -inf entries (and one row whose first 16
    # entries are all -inf): entropy equals scipy's entr (x log x with
    # entr(0) = 0) summed over the softmax, and the finite log-probs equal
    # those of the row with its masked columns removed.
    special = pytest.importorskip("scipy.special")
    g = torch.Generator().manual_seed(seed)
    seqs = [[1, 2, 3, 4, 5, 6]]
    pk = oracle.tree_pack(seqs, 128)
    V = 40
    logits = 2 * torch.randn((6, V), generator=g, dtype=torch.float64)
    masked = torch.rand((6, V), generator=g) < 0.3
    masked[:, 2] = False                                  # every label stays finite
    masked[:, 3:7] = False
    masked[0, :16] = True
    masked[0, 2] = False
    logits[masked] = float("-inf")
    lp, ent = oracle.sequence_logprobs_entropy(pk, seqs, logits, [0])
    p = torch.softmax(logits, -1).numpy()
    assert np.allclose(ent[0], special.entr(p).sum(-1), atol=1e-12)
    for t in range(5):
        keep = ~masked[t]
        sub = logits[t, keep]
        col = int(keep[:seqs[0][t + 1]].sum())            # label's column among the kept ones
        assert lp[0][t] == pytest.approx(float(torch.log_softmax(sub, -1)[col]), abs=1e-12)


@pytest.mark.parametrize("seed,hq,hkv,d", [(21, 4, 2, 16), (22, 2, 2, 8), (23, 6, 3, 8)])
def test_row_oracle_equals_node_oracle(seed, hq, hkv, d):
    # attn_rows (one query row at a time) against the node-level forward and
    # backward: O, LSE and dQ of every row, and dK/dV once every row is given
    seqs, pk, q, k, v, dO = _random_case(seed, hq, hkv, d, n=8)
    t = pk.trees[0]
    O, L = oracle.attn_forward(t, q[0], k[0], v[0], t_pad=128)
    dQ, dK, dV = oracle.attn_backward(t, q[0], k[0], v[0], dO[0], t_pad=128)
    rows = list(range(t.n))
    Or, Lr, dQr, dKr, dVr = oracle.attn_rows(t, q[0], k[0], v[0], rows, dO=dO[0])
    assert torch.allclose(Or, O[:t.n], atol=1e-12) and torch.allclose(Lr, L[:, :t.n], atol=1e-12)
    assert torch.allclose(dQr, dQ[:t.n], atol=1e-12)
    assert torch.allclose(dKr, dK, atol=1e-12) and torch.allclose(dVr, dV, atol=1e-12)
    # a subset of rows gives those rows' values unchanged
    sub = rows[::5]
    Os, Ls = oracle.attn_rows(t, q[0], k[0], v[0], sub)
    assert torch.allclose(Os, O[sub], atol=1e-12)
