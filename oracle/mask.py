"""Oracle ancestor mask and 128x128 block classes (test infrastructure).

The AReaL "树训练" page (§树构建过程 diagram) states the attention rule of a
packed tree: causal masking with tree structure, where a token attends only
to its ancestors (and, causally, to itself). §注意力机制 builds a block mask
with BLOCK_SIZE = 128 over the sequence padded to a multiple of the block
size, so that empty blocks are skipped.

Here the mask is built from the parent links alone (walking up from each
query), never from the subtree ends, and the block classes are obtained by
counting mask entries inside each 128x128 tile:
EMPTY = 0 entries, FULL = all 128*128 entries, PARTIAL = anything else.
"""
from __future__ import annotations

import numpy as np

from .pack import BLOCK_SIZE, OracleTree

EMPTY, PARTIAL, FULL = 0, 1, 2


def dense_mask(tree: OracleTree, t_pad: int | None = None) -> np.ndarray:
    """``M[i, j] = True`` iff flat position j is i or an ancestor of i.

    Built by walking ``parent`` from every query; positions >= n (padding) see
    nothing and are seen by nothing. Small trees only (O(T^2) memory)."""
    n = tree.n
    T = n if t_pad is None else t_pad
    M = np.zeros((T, T), dtype=bool)
    for i in range(n):
        j = i
        while j >= 0:
            M[i, j] = True
            j = int(tree.parent[j])
    return M


def ancestor_intervals(tree: OracleTree, i: int) -> list[tuple[int, int]]:
    """Inclusive flat ranges of the ancestors-or-self of position ``i``:
    the part of i's node up to i, then every ancestor node in full (walking
    the compressed nodes' parent links up to the root)."""
    nid = int(tree.node_id[i])
    out = [(int(tree.node_start[nid]), i)]
    nid = int(tree.node_parent[nid])
    while nid >= 0:
        out.append((int(tree.node_start[nid]), int(tree.node_end[nid])))
        nid = int(tree.node_parent[nid])
    return out


def _mask_rows(tree: OracleTree, r0: int, r1: int, t_pad: int) -> np.ndarray:
    rows = np.zeros((r1 - r0, t_pad), dtype=bool)
    for i in range(r0, min(r1, tree.n)):
        for a, b in ancestor_intervals(tree, i):
            rows[i - r0, a:b + 1] = True
    return rows


def block_classes(tree: OracleTree, t_pad: int) -> np.ndarray:
    """``[nblk, nblk]`` uint8 class of every (query block, key block) tile.

    Counts the ancestor mask over each tile, one 128-row slab at a time (the
    slab rows come from the node-level ancestor ranges, which equal the
    parent-walk mask; a test checks that on trees small enough for both)."""
    if t_pad % BLOCK_SIZE:
        raise ValueError("t_pad must be a multiple of 128")
    nblk = t_pad // BLOCK_SIZE
    cls = np.zeros((nblk, nblk), dtype=np.uint8)
    full = BLOCK_SIZE * BLOCK_SIZE
    for qb in range(nblk):
        q0 = qb * BLOCK_SIZE
        if q0 >= tree.n:
            break
        slab = _mask_rows(tree, q0, q0 + BLOCK_SIZE, t_pad)
        cnt = slab.reshape(BLOCK_SIZE, nblk, BLOCK_SIZE).sum(axis=(0, 2))
        cls[qb] = np.where(cnt == 0, EMPTY, np.where(cnt == full, FULL, PARTIAL))
    return cls


def block_classes_dense(M: np.ndarray) -> np.ndarray:
    """Block classes counted from a full dense mask (small trees)."""
    T = M.shape[0]
    nblk = T // BLOCK_SIZE
    cnt = M.reshape(nblk, BLOCK_SIZE, nblk, BLOCK_SIZE).sum(axis=(1, 3))
    full = BLOCK_SIZE * BLOCK_SIZE
    return np.where(cnt == 0, EMPTY, np.where(cnt == full, FULL, PARTIAL)).astype(np.uint8)


def block_csr(cls: np.ndarray) -> dict[str, np.ndarray]:
    """Non-empty tiles as two CSR lists.

    ``q_ptr/q_idx``: for each query block, its non-empty key blocks in
    ascending order; ``k_ptr/k_idx``: for each key block, its non-empty query
    blocks in ascending order. Each entry is ``2 * block + (class == FULL)``."""
    nblk = cls.shape[0]
    q_ptr, q_idx = [0], []
    for qb in range(nblk):
        for kb in range(nblk):
            if cls[qb, kb] != EMPTY:
                q_idx.append(2 * kb + int(cls[qb, kb] == FULL))
        q_ptr.append(len(q_idx))
    k_ptr, k_idx = [0], []
    for kb in range(nblk):
        for qb in range(nblk):
            if cls[qb, kb] != EMPTY:
                k_idx.append(2 * qb + int(cls[qb, kb] == FULL))
        k_ptr.append(len(k_idx))
    return {
        "q_ptr": np.array(q_ptr, np.int64), "q_idx": np.array(q_idx, np.int64),
        "k_ptr": np.array(k_ptr, np.int64), "k_idx": np.array(k_idx, np.int64),
    }


def ancestor_pairs(tree: OracleTree) -> int:
    """Number of (query, visible key) pairs: the sum over positions of
    depth + 1 (every query sees each of its ancestors and itself)."""
    return int(np.sum(tree.depth + 1))
