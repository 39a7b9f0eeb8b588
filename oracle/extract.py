"""Oracle sequence extraction (test infrastructure; see the package docstring).

Follows the AReaL "树训练" page, §树构建过程 step 1 (提取序列): the real
tokens of each sequence are read from the padded ``input_ids`` with the
``attention_mask``.

Reading (the page gives no more): the tokens of row r are the entries
input_ids[r, c] whose attention_mask[r, c] is non-zero, in column order, so
left padding, right padding and interior gaps are all handled; a row with no
such entry is an empty sequence, which packing rejects.
"""
from __future__ import annotations


def extract_sequences(input_ids, attention_mask) -> list[list[int]]:
    out = []
    for ids_row, mask_row in zip(input_ids, attention_mask):
        out.append([int(t) for t, m in zip(ids_row, mask_row) if int(m) != 0])
    return out
