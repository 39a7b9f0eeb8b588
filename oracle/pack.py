"""Oracle trie packer (test infrastructure; see the package docstring).

Follows the AReaL "树训练" page, §树构建过程 (tree building):

  step 2 (贪心打包)  sequences are inserted into a trie greedily with a
                     first-fit-decreasing policy; a tree is one micro-batch and
                     holds at most ``max_tokens_per_mb`` tokens (§配置 table:
                     "每棵树的最大 token 数"), which must be a multiple of
                     BLOCK_SIZE = 128 (§配置 note);
  step 3 (Trie 压缩) linear chains are merged into single compressed nodes;

and §数据结构 ``TrieNode``: nodes carry inclusive ``[start_idx, end_idx]``
ranges into the flattened tree, children are keyed by their branching token,
and the root lists all nodes in preorder.

Readings taken where the page is silent (each is a fixed rule here):
  * "decreasing" orders by sequence length, longest first; equal lengths keep
    their input order (stable sort);
  * "first fit" tries the trees in creation order and takes the first whose
    token count plus the sequence's NEW (not already shared) tokens fits;
  * a node starts at a trie vertex whose parent is the root or has a child
    count other than one, and extends while the current vertex has exactly one
    child (a sequence may end inside a node);
  * children are visited in insertion order (the order the first sequence
    that created them arrived), both for the preorder layout and for nodes;
  * empty sequences and sequences longer than ``max_tokens_per_mb`` are
    rejected.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 128


class PackError(ValueError):
    """Invalid packing input; ``code`` names the condition."""

    def __init__(self, code: str, msg: str):
        super().__init__(f"{code}: {msg}")
        self.code = code


class _Trie:
    """Uncompressed token trie. Vertex 0 is the root; every other vertex holds
    one token. ``children[v]`` is a dict token -> vertex in insertion order."""

    def __init__(self) -> None:
        self.token: list[int] = [-1]
        self.parent: list[int] = [-1]
        self.children: list[dict[int, int]] = [{}]

    @property
    def n_tokens(self) -> int:
        return len(self.token) - 1

    def shared_prefix(self, seq: list[int]) -> int:
        v, n = 0, 0
        for t in seq:
            nxt = self.children[v].get(t)
            if nxt is None:
                break
            v, n = nxt, n + 1
        return n

    def insert(self, seq: list[int]) -> list[int]:
        """Insert ``seq``; return the vertex of each of its tokens."""
        path, v = [], 0
        for t in seq:
            nxt = self.children[v].get(t)
            if nxt is None:
                nxt = len(self.token)
                self.token.append(t)
                self.parent.append(v)
                self.children.append({})
                self.children[v][t] = nxt
            path.append(nxt)
            v = nxt
        return path


@dataclass
class OracleTree:
    """One packed tree (= one micro-batch) in flattened preorder."""

    seq_ids: list[int]
    tokens: np.ndarray        # [n] token id at each flat position
    parent: np.ndarray        # [n] flat position of the parent token, -1 at root children
    depth: np.ndarray         # [n] number of ancestors (= position id inside any sequence)
    subtree_end: np.ndarray   # [n] last flat position of the subtree of the token's node
    node_id: np.ndarray       # [n] compressed node holding each position
    node_start: np.ndarray    # [N] inclusive flat range of each compressed node ...
    node_end: np.ndarray      # [N] ... (nodes listed in preorder)
    node_parent: np.ndarray   # [N] parent node, -1 under the root
    node_subtree_end: np.ndarray  # [N]

    @property
    def n(self) -> int:
        return int(self.tokens.shape[0])

    def children_of(self, pos: int) -> list[int]:
        """Flat positions whose parent is ``pos``, in flat order."""
        return [int(c) for c in np.nonzero(self.parent == pos)[0]]


@dataclass
class OraclePacking:
    max_tokens_per_mb: int
    trees: list[OracleTree]
    seq_tree: np.ndarray              # [n_seqs] tree holding each input sequence
    seq_pos: list[np.ndarray] = field(default_factory=list)  # per sequence: flat positions
    total_seq_tokens: int = 0

    @property
    def n_trees(self) -> int:
        return len(self.trees)

    @property
    def total_tree_tokens(self) -> int:
        return sum(t.n for t in self.trees)

    @property
    def tree_token_ratio(self) -> float:
        """Tree tokens over original tokens (§指标和监控 ``tree_token_ratio``)."""
        return self.total_tree_tokens / self.total_seq_tokens


def _validate(seqs: list[list[int]], mb: int) -> None:
    if mb <= 0 or mb % BLOCK_SIZE != 0:
        raise PackError("INVALID_ARG", f"max_tokens_per_mb={mb} must be a positive multiple of {BLOCK_SIZE}")
    if len(seqs) == 0:
        raise PackError("INVALID_ARG", "no sequences")
    for s, seq in enumerate(seqs):
        if len(seq) == 0:
            raise PackError("EMPTY_SEQUENCE", f"sequence {s} is empty")
        if len(seq) > mb:
            raise PackError("SEQ_TOO_LONG", f"sequence {s} has {len(seq)} tokens > {mb}")
        if any(t < 0 for t in seq):
            raise PackError("INVALID_ARG", f"sequence {s} holds a negative token id")


def _flatten(trie: _Trie, seq_ids: list[int]) -> tuple[OracleTree, np.ndarray]:
    """Preorder layout of ``trie``; returns the tree and vertex -> position."""
    nv = len(trie.token)
    pos = np.full(nv, -1, dtype=np.int64)
    order: list[int] = []
    stack = list(reversed(list(trie.children[0].values())))
    while stack:
        v = stack.pop()
        pos[v] = len(order)
        order.append(v)
        stack.extend(reversed(list(trie.children[v].values())))
    n = len(order)
    tokens = np.array([trie.token[v] for v in order], dtype=np.int64)
    parent = np.array([pos[trie.parent[v]] if trie.parent[v] != 0 else -1 for v in order], dtype=np.int64)
    depth = np.zeros(n, dtype=np.int64)
    for p in range(n):                        # parents precede children in preorder
        depth[p] = 0 if parent[p] < 0 else depth[parent[p]] + 1
    size = np.ones(n, dtype=np.int64)
    for p in range(n - 1, -1, -1):            # children follow parents in preorder
        if parent[p] >= 0:
            size[parent[p]] += size[p]
    subtree_end = np.arange(n, dtype=np.int64) + size - 1

    # Linear-chain compression (§树构建过程 step 3).
    node_start, node_end, node_parent = [], [], []
    node_id = np.full(n, -1, dtype=np.int64)
    for p, v in enumerate(order):
        pv = trie.parent[v]
        if pv != 0 and len(trie.children[pv]) == 1:
            continue                          # v continues its parent's chain
        nid = len(node_start)
        cur = v
        while True:
            node_id[pos[cur]] = nid
            if len(trie.children[cur]) != 1:
                break
            cur = next(iter(trie.children[cur].values()))
        node_start.append(p)
        node_end.append(int(pos[cur]))
        node_parent.append(-1 if pv == 0 else int(node_id[pos[pv]]))
    node_start = np.array(node_start, dtype=np.int64)
    node_end = np.array(node_end, dtype=np.int64)
    tree = OracleTree(
        seq_ids=seq_ids, tokens=tokens, parent=parent, depth=depth,
        subtree_end=subtree_end[node_start[node_id]] if n else subtree_end,
        node_id=node_id, node_start=node_start, node_end=node_end,
        node_parent=np.array(node_parent, dtype=np.int64),
        node_subtree_end=subtree_end[node_start] if n else node_start,
    )
    return tree, pos


def tree_pack(seqs: list[list[int]], max_tokens_per_mb: int) -> OraclePacking:
    """Pack ``seqs`` into prefix tries of at most ``max_tokens_per_mb`` tokens."""
    seqs = [list(map(int, s)) for s in seqs]
    _validate(seqs, max_tokens_per_mb)
    order = sorted(range(len(seqs)), key=lambda s: -len(seqs[s]))   # stable
    tries: list[_Trie] = []
    members: list[list[int]] = []
    paths: dict[int, tuple[int, list[int]]] = {}
    for s in order:
        seq = seqs[s]
        for b, trie in enumerate(tries):
            new = len(seq) - trie.shared_prefix(seq)
            if trie.n_tokens + new <= max_tokens_per_mb:
                break
        else:
            tries.append(_Trie())
            members.append([])
            b = len(tries) - 1
        paths[s] = (b, tries[b].insert(seq))
        members[b].append(s)
    trees, vpos = [], []
    for b, trie in enumerate(tries):
        tree, pos = _flatten(trie, members[b])
        trees.append(tree)
        vpos.append(pos)
    seq_tree = np.array([paths[s][0] for s in range(len(seqs))], dtype=np.int64)
    seq_pos = [vpos[paths[s][0]][np.array(paths[s][1], dtype=np.int64)] for s in range(len(seqs))]
    return OraclePacking(max_tokens_per_mb, trees, seq_tree, seq_pos,
                         total_seq_tokens=sum(len(s) for s in seqs))


def padded_arrays(pk: OraclePacking) -> dict[str, np.ndarray]:
    """The per-tree arrays padded to ``[B, T_pad]`` with the layout's pad
    values (token/subtree_end/parent/node_id -1, depth 0), for comparison with
    the library's flat metadata."""
    B, T = pk.n_trees, pk.max_tokens_per_mb
    out = {
        "tokens": np.full((B, T), -1, np.int64),
        "subtree_end": np.full((B, T), -1, np.int64),
        "parent": np.full((B, T), -1, np.int64),
        "depth": np.zeros((B, T), np.int64),
        "node_id": np.full((B, T), -1, np.int64),
        "n_tokens": np.array([t.n for t in pk.trees], np.int64),
    }
    for b, t in enumerate(pk.trees):
        for k in ("tokens", "subtree_end", "parent", "depth", "node_id"):
            out[k][b, : t.n] = getattr(t, k)
    return out
