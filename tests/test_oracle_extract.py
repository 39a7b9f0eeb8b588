"""Pins for the oracle sequence extraction (tree training page, §树构建过程
step 1: real tokens come from input_ids with attention_mask), including the
page's worked example recovered from a padded batch."""
import oracle
from oracle.extract import extract_sequences

A, B, C, D, E, F, G, H = range(8)


def test_right_left_and_interior_padding():
    ids = [[5, 6, 7, 0, 0], [0, 0, 8, 9, 1], [2, 0, 3, 0, 4]]
    mask = [[1, 1, 1, 0, 0], [0, 0, 1, 1, 1], [1, 0, 1, 0, 1]]
    assert extract_sequences(ids, mask) == [[5, 6, 7], [8, 9, 1], [2, 3, 4]]


def test_pad_ids_never_leak():
    # a pad id equal to a real token id is still dropped by the mask
    assert extract_sequences([[7, 7, 7]], [[0, 1, 0]]) == [[7]]


def test_worked_example_from_a_padded_batch():
    # the page's three sequences, right-padded to 4 with id 0 (= token A!)
    ids = [[A, B, C, D], [A, B, E, F], [A, G, H, A]]
    mask = [[1, 1, 1, 1], [1, 1, 1, 1], [1, 1, 1, 0]]
    seqs = extract_sequences(ids, mask)
    assert seqs == [[A, B, C, D], [A, B, E, F], [A, G, H]]
    pk = oracle.tree_pack(seqs, 128)
    assert pk.trees[0].n == 8 and pk.total_seq_tokens == 11


def test_empty_row_extracts_empty():
    assert extract_sequences([[1, 2]], [[0, 0]]) == [[]]
