"""Oracle fp64 tree attention, forward and backward (test infrastructure).

Semantics from the AReaL "树训练" page: §树构建过程's diagram gives the mask
(causal, with tree structure: a token attends only to its ancestors and
itself); §注意力机制 computes masked softmax attention over the packed tree.
The pages leave the scale and head grouping open; the readings here are the
usual ones: scores ``q.k * scale`` with ``scale = 1/sqrt(d)`` unless given,
and grouped-query attention where query head h reads key/value head
``h // (Hq // Hkv)``.

For query position i with ancestor-or-self set A(i):

    S_ij = scale * q_i . k_j,           j in A(i)
    LSE_i = log sum_{j in A(i)} exp(S_ij)
    O_i   = sum_{j in A(i)} exp(S_ij - LSE_i) v_j

and for an upstream gradient dO the exact gradient of <dO, O>:

    P_ij = exp(S_ij - LSE_i),   D_i = dO_i . O_i
    dV_j += P_ij dO_i,          dS_ij = P_ij (dO_i . v_j - D_i)
    dQ_i = scale sum_j dS_ij k_j,   dK_j += scale dS_ij q_i

(dK, dV summed over the query heads that share a key/value head). Padding
rows give O = 0, LSE = 0 and zero gradients.  ``attn_rows`` computes the same
quantities one query row at a time, for trees too large for the node-level
functions (a 131072-token chain); it is pinned against them on small trees.

Computation is organised node by node: the queries of one compressed node
share their root path, so A(i) is a prefix of that path (all ancestor nodes'
tokens, then the node's own tokens up to i). Everything is fp64 on the exact
(bf16-representable) input values.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from .pack import OracleTree

_CHUNK = 256   # query rows per block of work (memory bound only; no reordering of sums)


def _root_path(tree: OracleTree, nid: int) -> np.ndarray:
    """Flat positions from the root down to the end of node ``nid``."""
    chain = []
    while nid >= 0:
        chain.append(nid)
        nid = int(tree.node_parent[nid])
    parts = [np.arange(tree.node_start[c], tree.node_end[c] + 1) for c in reversed(chain)]
    return np.concatenate(parts)


def _as64(x: torch.Tensor) -> torch.Tensor:
    return x.detach().to("cpu").to(torch.float64)


def attn_forward(tree: OracleTree, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                 scale: float | None = None, t_pad: int | None = None,
                 nodes: list[int] | None = None):
    """fp64 forward for one tree.

    q ``[T, Hq, d]``, k/v ``[T, Hkv, d]`` (any float dtype; widened to fp64).
    Returns O ``[T, Hq, d]`` and LSE ``[Hq, T]`` fp64 (pad rows 0). ``nodes``
    restricts the work to those compressed nodes (rows elsewhere stay 0)."""
    T = q.shape[0] if t_pad is None else t_pad
    Hq, d = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    q64, k64, v64 = _as64(q), _as64(k), _as64(v)
    O = torch.zeros((T, Hq, d), dtype=torch.float64)
    LSE = torch.zeros((Hq, T), dtype=torch.float64)
    node_list = range(len(tree.node_start)) if nodes is None else nodes
    for nid in node_list:
        path = torch.from_numpy(_root_path(tree, nid))
        s0, s1 = int(tree.node_start[nid]), int(tree.node_end[nid])
        base = path.numel() - (s1 - s0 + 1)
        kp = k64[path].repeat_interleave(G, dim=1)        # [P, Hq, d]
        vp = v64[path].repeat_interleave(G, dim=1)
        for c0 in range(s0, s1 + 1, _CHUNK):
            c1 = min(s1 + 1, c0 + _CHUNK)
            qi = q64[c0:c1]                                # [m, Hq, d]
            S = torch.einsum("mhd,phd->hmp", qi, kp) * scale
            rows = torch.arange(c0 - s0, c1 - s0) + base   # path index of each query
            allowed = torch.arange(path.numel())[None, :] <= rows[:, None]
            S = S.masked_fill(~allowed[None], float("-inf"))
            lse = torch.logsumexp(S, dim=-1)               # [Hq, m]
            P = torch.exp(S - lse[..., None])
            O[c0:c1] = torch.einsum("hmp,phd->mhd", P, vp)
            LSE[:, c0:c1] = lse
    return O, LSE


def attn_backward(tree: OracleTree, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                  dO: torch.Tensor, scale: float | None = None, t_pad: int | None = None,
                  nodes: list[int] | None = None):
    """fp64 gradients (dQ, dK, dV) of ``<dO, O>`` for one tree.

    Uses the fp64 forward's own O and LSE. ``nodes`` restricts the QUERY
    nodes whose contributions are accumulated (dK/dV then hold only those
    contributions; dQ rows of other nodes stay 0)."""
    T = q.shape[0] if t_pad is None else t_pad
    Hq, d = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    q64, k64, v64, do64 = _as64(q), _as64(k), _as64(v), _as64(dO)
    dQ = torch.zeros((T, Hq, d), dtype=torch.float64)
    dKh = torch.zeros((T, Hq, d), dtype=torch.float64)   # per query head, summed per group below
    dVh = torch.zeros((T, Hq, d), dtype=torch.float64)
    node_list = range(len(tree.node_start)) if nodes is None else nodes
    for nid in node_list:
        path = torch.from_numpy(_root_path(tree, nid))
        s0, s1 = int(tree.node_start[nid]), int(tree.node_end[nid])
        base = path.numel() - (s1 - s0 + 1)
        kp = k64[path].repeat_interleave(G, dim=1)
        vp = v64[path].repeat_interleave(G, dim=1)
        for c0 in range(s0, s1 + 1, _CHUNK):
            c1 = min(s1 + 1, c0 + _CHUNK)
            qi, doi = q64[c0:c1], do64[c0:c1]
            S = torch.einsum("mhd,phd->hmp", qi, kp) * scale
            rows = torch.arange(c0 - s0, c1 - s0) + base
            allowed = torch.arange(path.numel())[None, :] <= rows[:, None]
            S = S.masked_fill(~allowed[None], float("-inf"))
            lse = torch.logsumexp(S, dim=-1)
            P = torch.exp(S - lse[..., None])              # [Hq, m, P]
            Oi = torch.einsum("hmp,phd->mhd", P, vp)
            Di = (doi * Oi).sum(-1).transpose(0, 1)         # [Hq, m]
            dP = torch.einsum("mhd,phd->hmp", doi, vp)
            dS = P * (dP - Di[..., None])
            dQ[c0:c1] = scale * torch.einsum("hmp,phd->mhd", dS, kp)
            dKh.index_add_(0, path, scale * torch.einsum("hmp,mhd->phd", dS, qi))
            dVh.index_add_(0, path, torch.einsum("hmp,mhd->phd", P, doi))
    dK = dKh.view(T, Hkv, G, d).sum(2)
    dV = dVh.view(T, Hkv, G, d).sum(2)
    return dQ, dK, dV


def _ancestors_of(tree: OracleTree, i: int) -> np.ndarray:
    """Positions query i sees, in ascending order: the tokens of every
    ancestor node of node(i), then node(i)'s own tokens up to i."""
    nid = int(tree.node_id[i])
    path = _root_path(tree, nid)
    return path[path <= i] if path.size and path[-1] > i else path


def attn_rows(tree: OracleTree, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, rows,
              dO: torch.Tensor | None = None, scale: float | None = None):
    """fp64 attention of selected query positions, one row at a time (for
    trees too large for the node-level functions above).

    Returns O ``[len(rows), Hq, d]`` and LSE ``[Hq, len(rows)]``; with ``dO``
    also dQ of those rows ``[len(rows), Hq, d]`` and the contributions of
    those query rows to dK and dV ``[T, Hkv, d]`` (summed over the query heads
    of each key/value head).  When ``rows`` holds every query that sees a
    key, that key's dK/dV rows are complete."""
    T = q.shape[0]
    Hq, d = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    rows = [int(r) for r in rows]
    k64, v64 = _as64(k), _as64(v)
    O = torch.zeros((len(rows), Hq, d), dtype=torch.float64)
    LSE = torch.zeros((Hq, len(rows)), dtype=torch.float64)
    dQ = torch.zeros((len(rows), Hq, d), dtype=torch.float64)
    dK = torch.zeros((T, Hkv, d), dtype=torch.float64)
    dV = torch.zeros((T, Hkv, d), dtype=torch.float64)
    for u, i in enumerate(rows):
        if i >= tree.n:
            continue
        anc = torch.from_numpy(_ancestors_of(tree, i))
        qi = _as64(q[i]).view(Hkv, G, d)                          # query heads of each kv head
        kp, vp = k64[anc], v64[anc]                               # [P, Hkv, d]
        S = torch.einsum("hgd,phd->hgp", qi, kp) * scale
        lse = torch.logsumexp(S, dim=-1)
        P = torch.exp(S - lse[..., None])                         # [Hkv, G, P]
        Oi = torch.einsum("hgp,phd->hgd", P, vp)
        O[u] = Oi.reshape(Hq, d)
        LSE[:, u] = lse.reshape(Hq)
        if dO is None:
            continue
        doi = _as64(dO[i]).view(Hkv, G, d)
        Di = (doi * Oi).sum(-1)                                    # [Hkv, G]
        dP = torch.einsum("hgd,phd->hgp", doi, vp)
        dS = P * (dP - Di[..., None])
        dQ[u] = (scale * torch.einsum("hgp,phd->hgd", dS, kp)).reshape(Hq, d)
        dK.index_add_(0, anc, scale * torch.einsum("hgp,hgd->phd", dS, qi))
        dV.index_add_(0, anc, torch.einsum("hgp,hgd->phd", P, doi))
    if dO is None:
        return O, LSE
    return O, LSE, dQ, dK, dV
