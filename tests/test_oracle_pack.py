"""Pins for the oracle packer (CPU).

Each check rests on something fixed outside the packer's own code: the tree
training page's worked example (tests/golden/worked_example.json), closed
forms (tree tokens = distinct non-empty prefixes), brute force over tiny
random inputs, and hand cases for the first-fit-decreasing rule.
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle.mask import dense_mask
from oracle.pack import PackError, padded_arrays
from synth import make_sequences, random_small_sequences, CONFIGS

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")


def _prefix_count(seqs):
    return len({tuple(s[:i]) for s in seqs for i in range(1, len(s) + 1)})


def test_worked_example_counts_and_shape():
    g = json.load(open(GOLDEN))
    pk = oracle.tree_pack(g["sequences"], 128)
    assert pk.n_trees == 1
    t = pk.trees[0]
    assert pk.total_seq_tokens == g["original_tokens"]
    assert t.n == g["tree_tokens"]
    assert pk.tree_token_ratio == pytest.approx(8 / 11)
    letters = g["letters"]
    # every drawn edge child -> parent appears, and nothing else
    edges = {}
    for p in range(t.n):
        if t.parent[p] >= 0:
            edges[letters[t.tokens[p]]] = letters[t.tokens[t.parent[p]]]
    assert edges == g["tree_edges_child_to_parent"]
    roots = [letters[t.tokens[p]] for p in range(t.n) if t.parent[p] < 0]
    assert roots == g["tree_roots"]
    nodes = ["".join(letters[t.tokens[p]] for p in range(s, e + 1))
             for s, e in zip(t.node_start, t.node_end)]
    assert sorted(nodes) == sorted(g["compressed_nodes_letters"])


def test_worked_example_layout_under_readings():
    # Preorder with children in insertion order gives A B C D E F G H.
    g = json.load(open(GOLDEN))
    t = oracle.tree_pack(g["sequences"], 128).trees[0]
    assert t.tokens.tolist() == list(range(8))
    assert t.subtree_end.tolist() == [7, 5, 3, 3, 5, 5, 7, 7]
    assert list(zip(t.node_start.tolist(), t.node_end.tolist())) == [(0, 0), (1, 1), (2, 3), (4, 5), (6, 7)]
    assert t.node_parent.tolist() == [-1, 0, 1, 1, 0]
    assert t.depth.tolist() == [0, 1, 2, 3, 2, 3, 1, 2]


def _check_invariants(seqs, pk):
    mb = pk.max_tokens_per_mb
    for b, t in enumerate(pk.trees):
        assert t.n <= mb
        mem = [seqs[s] for s in t.seq_ids]
        assert t.n == _prefix_count(mem)                       # closed form
        assert np.all(t.parent < np.arange(t.n))                 # preorder: parents first
        M = dense_mask(t)
        E = t.subtree_end
        i = np.arange(t.n)[:, None]
        j = np.arange(t.n)[None, :]
        assert np.array_equal(M, (j <= i) & (i <= E[None, :]))   # interval form of the mask
        assert np.array_equal(M.sum(1), t.depth + 1)
        # compressed nodes: contiguous, tile the tree, split exactly at branchings
        nchild = np.bincount(t.parent[t.parent >= 0], minlength=t.n)
        starts = [p for p in range(t.n) if t.parent[p] < 0 or nchild[t.parent[p]] != 1]
        assert t.node_start.tolist() == starts
        for nid, (s, e) in enumerate(zip(t.node_start, t.node_end)):
            assert np.all(t.node_id[s:e + 1] == nid)
            assert all(nchild[p] == 1 for p in range(s, e))
            assert nchild[e] != 1
            par = t.parent[s]
            assert t.node_parent[nid] == (-1 if par < 0 else t.node_id[par])
    # every sequence is recovered in order from its positions
    for s, seq in enumerate(seqs):
        t = pk.trees[pk.seq_tree[s]]
        pos = pk.seq_pos[s]
        assert t.tokens[pos].tolist() == list(seq)
        assert t.depth[pos].tolist() == list(range(len(seq)))
        assert t.parent[pos[0]] == -1
        assert np.array_equal(t.parent[pos[1:]], pos[:-1])
        assert s in t.seq_ids


@pytest.mark.parametrize("seed", range(40))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(seed)
    seqs = random_small_sequences(rng, int(rng.integers(1, 9)), 12, int(rng.integers(2, 5)))
    mb = 128 * int(rng.integers(1, 3))
    pk = oracle.tree_pack(seqs, mb)
    _check_invariants(seqs, pk)
    assert pk.total_tree_tokens == sum(_prefix_count([seqs[s] for s in t.seq_ids]) for t in pk.trees)


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_multi_tree(seed):
    # long sequences over a tiny vocabulary with mb = 128: several trees
    rng = np.random.default_rng(100 + seed)
    seqs = random_small_sequences(rng, 12, 100, 3, min_len=20)
    pk = oracle.tree_pack(seqs, 128)
    assert pk.n_trees >= 2
    _check_invariants(seqs, pk)


def test_first_fit_uses_creation_order():
    # lengths 100, 50, 20 of disjoint tokens, mb = 128: the 20 goes into the
    # FIRST tree with room (tree 0, 120 tokens), not the lightest (tree 1)
    a = [1] + [5] * 99
    b = [2] + [6] * 49
    c = [3] + [7] * 19
    pk = oracle.tree_pack([c, a, b], 128)
    assert pk.n_trees == 2
    assert pk.trees[0].seq_ids == [1, 0] and pk.trees[0].n == 120
    assert pk.trees[1].seq_ids == [2] and pk.trees[1].n == 50


def test_fit_counts_only_new_tokens():
    base = list(range(1, 101))
    s1 = base + [500 + i for i in range(28)]           # 128 tokens
    s2 = base + [900 + i for i in range(20)]           # 120 tokens, 100 shared -> 20 new
    pk = oracle.tree_pack([s1, s2], 128)               # 128 + 20 > 128: second tree
    assert pk.n_trees == 2
    pk = oracle.tree_pack([s1, s2], 256)
    assert pk.n_trees == 1 and pk.trees[0].n == 148
    pk = oracle.tree_pack([s1, list(s1), s1[:50]], 128)  # duplicates add nothing
    assert pk.n_trees == 1 and pk.trees[0].n == 128


def test_stable_order_on_equal_lengths():
    seqs = [[9, 1], [8, 2], [9, 3], [7]]
    t = oracle.tree_pack(seqs, 128).trees[0]
    assert t.seq_ids == [0, 1, 2, 3]
    assert t.tokens.tolist() == [9, 1, 3, 8, 2, 7]   # children of 9 in insertion order


def test_special_cases():
    one = oracle.tree_pack([[4, 5, 6, 7]], 128)
    assert one.tree_token_ratio == 1.0 and len(one.trees[0].node_start) == 1
    same = oracle.tree_pack([[4, 5, 6]] * 5, 128)
    assert same.tree_token_ratio == pytest.approx(1 / 5)
    disjoint = oracle.tree_pack([[1, 2], [3, 4], [5]], 128)
    t = disjoint.trees[0]
    assert disjoint.tree_token_ratio == 1.0
    assert int(np.sum(t.parent < 0)) == 3 and len(t.node_start) == 3
    ends_mid_chain = oracle.tree_pack([[1, 2, 3], [1, 2]], 128).trees[0]
    assert len(ends_mid_chain.node_start) == 1          # [1,2] ends inside the node


def test_errors():
    with pytest.raises(PackError) as e:
        oracle.tree_pack([[1]], 100)
    assert e.value.code == "INVALID_ARG"
    with pytest.raises(PackError) as e:
        oracle.tree_pack([[1], []], 128)
    assert e.value.code == "EMPTY_SEQUENCE"
    with pytest.raises(PackError) as e:
        oracle.tree_pack([[1] * 129], 128)
    assert e.value.code == "SEQ_TOO_LONG"
    with pytest.raises(PackError):
        oracle.tree_pack([], 128)
    with pytest.raises(PackError):
        oracle.tree_pack([[1, -2]], 128)


@pytest.mark.parametrize("cid", [1, 2, 3, 5])
def test_workloads_pack(cid):
    seqs = make_sequences(cid)
    cfg = CONFIGS[cid]
    pk = oracle.tree_pack(seqs, cfg.max_tokens_per_mb)
    assert all(t.n <= cfg.max_tokens_per_mb for t in pk.trees)
    assert pk.tree_token_ratio < 1.0
    for s, seq in enumerate(seqs):
        t = pk.trees[pk.seq_tree[s]]
        assert t.tokens[pk.seq_pos[s]].tolist() == seq
    arr = padded_arrays(pk)
    assert arr["tokens"].shape == (pk.n_trees, cfg.max_tokens_per_mb)
