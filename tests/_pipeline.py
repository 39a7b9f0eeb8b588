"""Shared helpers of the GPU parity tests: run the library path on seeded
inputs and compare against the oracle with the stated tolerances."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from synth import CONFIGS, make_dout, make_qkv, make_sequences

ATTN_MAX_ABS = 2e-2   # attention outputs and gradients vs fp64
ATTN_REL_L2 = 5e-3
LOGP_ABS = 1e-3       # log-probs and entropies vs fp64


def assert_attn_close(got: torch.Tensor, ref: torch.Tensor, what: str,
                      max_abs: float = ATTN_MAX_ABS, rel_l2: float = ATTN_REL_L2) -> tuple[float, float]:
    g = got.detach().to("cpu", torch.float64)
    r = ref.detach().to("cpu", torch.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert torch.isfinite(g).all(), f"{what}: non-finite values"
    err = (g - r).abs().max().item() if g.numel() else 0.0
    nrm = r.norm().item()
    rel = (g - r).norm().item() / nrm if nrm > 0 else (g - r).norm().item()
    assert err <= max_abs and rel <= rel_l2, f"{what}: max-abs {err:.3e}, rel-L2 {rel:.3e}"
    return err, rel


def bf16_half_ulp(x: torch.Tensor) -> torch.Tensor:
    """Half the bf16 spacing at |x|: the least error any bf16 output of x has."""
    ax = x.abs().clamp_min(2.0 ** -126)
    return torch.exp2(torch.floor(torch.log2(ax)) - 8)


def assert_attn_close_bf16_out(got: torch.Tensor, ref: torch.Tensor, what: str) -> None:
    """Bound for bf16-valued outputs: the stated max-abs plus the rounding to
    bf16 that the output type itself forces, element by element."""
    g = got.detach().to("cpu", torch.float64)
    r = ref.detach().to("cpu", torch.float64)
    assert torch.isfinite(g).all(), f"{what}: non-finite values"
    excess = ((g - r).abs() - (ATTN_MAX_ABS + bf16_half_ulp(r))).max().item()
    rel = (g - r).norm().item() / max(r.norm().item(), 1e-30)
    assert excess <= 0 and rel <= ATTN_REL_L2, f"{what}: excess {excess:.3e}, rel-L2 {rel:.3e}"


# Canary guard bands: an output buffer is allocated with GUARD elements on
# each side holding a fixed bit pattern, the call writes the interior view,
# and check_guards() verifies afterwards that no kernel wrote past either end.
GUARD = 4096
_PATTERN = {1: (torch.uint8, 0xA5), 2: (torch.int16, 0x7FA5), 4: (torch.int32, 0x7FA5A5A5)}


def guarded(shape, dtype, device="cuda"):
    """(backing buffer, interior view of ``shape``) with canaries on both sides."""
    n = 1
    for x in shape:
        n *= int(x)
    buf = torch.empty(n + 2 * GUARD, dtype=dtype, device=device)
    ity, pat = _PATTERN[buf.element_size()]
    buf.view(ity).fill_(pat)
    return buf, buf[GUARD:GUARD + n].view(tuple(shape))


def check_guards(buf: torch.Tensor, what: str) -> None:
    ity, pat = _PATTERN[buf.element_size()]
    raw = buf.view(ity)
    assert torch.all(raw[:GUARD] == pat) and torch.all(raw[-GUARD:] == pat), f"{what}: write outside the buffer"


def bf16_operand_bounds(tree, q, k, v, dO, t_pad: int):
    """Per-element bounds on the gradient error that the backward's bf16
    roundings alone cause, as FlashAttention-style kernels have them: the
    tensor cores take P (for dV) and dS (for dQ and dK) as bf16 operands, and
    D = rowsum(dO * O) is formed from the bf16 O the forward returned.
    Rounding to bf16 changes a value by at most 2^-8 of it; with u = 2^-7
    (twice that, for margin):
        e_D_i  = u sum_d |dO_id| |O_id|,   e_dS_ij = u |dS_ij| + P_ij e_D_i
        dQ_i: scale sum_j e_dS_ij |k_j|,  dK_j: scale sum_i e_dS_ij |q_i|,
        dV_j: u sum_i P_ij |dO_i|,
    from the fp64 reference's own P, dS and O.  Returns (bq [T,Hq,d], bk, bv [T,Hkv,d])."""
    from oracle.attention import _root_path
    Hq, d = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    G = Hq // Hkv
    sc = 1.0 / math.sqrt(d)
    u = 2.0 ** -7
    q64, k64, v64, do64 = (x.detach().to("cpu", torch.float64) for x in (q, k, v, dO))
    bq = torch.zeros((t_pad, Hq, d), dtype=torch.float64)
    bkh = torch.zeros((t_pad, Hq, d), dtype=torch.float64)
    bvh = torch.zeros((t_pad, Hq, d), dtype=torch.float64)
    for nid in range(len(tree.node_start)):
        path = torch.from_numpy(_root_path(tree, nid))
        s0, s1 = int(tree.node_start[nid]), int(tree.node_end[nid])
        base = path.numel() - (s1 - s0 + 1)
        kp, vp = k64[path].repeat_interleave(G, 1), v64[path].repeat_interleave(G, 1)
        qi, doi = q64[s0:s1 + 1], do64[s0:s1 + 1]
        S = torch.einsum("mhd,phd->hmp", qi, kp) * sc
        rows = torch.arange(s1 - s0 + 1) + base
        S = S.masked_fill(~(torch.arange(path.numel())[None, :] <= rows[:, None])[None], float("-inf"))
        P = torch.softmax(S, -1)
        Oi = torch.einsum("hmp,phd->mhd", P, vp)
        Di = (doi * Oi).sum(-1).transpose(0, 1)                           # [Hq, m]
        eD = u * (doi.abs() * Oi.abs()).sum(-1).transpose(0, 1)            # [Hq, m]
        dS = P * (torch.einsum("mhd,phd->hmp", doi, vp) - Di[..., None])
        edS = u * dS.abs() + P * eD[..., None]
        bq[s0:s1 + 1] = sc * torch.einsum("hmp,phd->mhd", edS, kp.abs())
        bkh.index_add_(0, path, sc * torch.einsum("hmp,mhd->phd", edS, qi.abs()))
        bvh.index_add_(0, path, u * torch.einsum("hmp,mhd->phd", P, doi.abs()))
    return bq, bkh.view(t_pad, Hkv, G, d).sum(2), bvh.view(t_pad, Hkv, G, d).sum(2)


def assert_grad_close_with_operand_rounding(got, ref, bound, what):
    """max-abs 2e-2 plus the bf16-rounding bound, element by element; rel-L2 5e-3."""
    g = got.detach().to("cpu", torch.float64)
    r = ref.detach().to("cpu", torch.float64)
    assert torch.isfinite(g).all(), f"{what}: non-finite values"
    excess = ((g - r).abs() - (ATTN_MAX_ABS + bound)).max().item()
    rel = (g - r).norm().item() / max(r.norm().item(), 1e-30)
    assert excess <= 0 and rel <= ATTN_REL_L2, f"{what}: excess {excess:.3e}, rel-L2 {rel:.3e}"


def pack_and_upload(tpa, seqs, mb, device="cuda"):
    tree = tpa.tree_pack(seqs, mb)
    dtree = tree.upload(device)
    mask = tpa.block_classify(dtree)
    return tree, dtree, mask


def random_inputs(B, T, hq, hkv, d, seed, device="cuda"):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, T, hq, d), generator=g).to(torch.bfloat16)
    k = torch.randn((B, T, hkv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, T, hkv, d), generator=g).to(torch.bfloat16)
    do = torch.randn((B, T, hq, d), generator=g).to(torch.bfloat16)
    return [x.to(device) for x in (q, k, v, do)], (q, k, v, do)


def workload(cid: int):
    cfg = CONFIGS[cid]
    seqs = make_sequences(cid)
    return cfg, seqs


def workload_tensors(cid: int, B: int, T: int):
    cfg = CONFIGS[cid]
    q, k, v = make_qkv(cid, B, T, cfg.n_heads_q, cfg.n_heads_kv, cfg.head_dim)
    do = make_dout(cid, B, T, cfg.n_heads_q, cfg.head_dim)
    return q, k, v, do


def leaf_nodes(tree: oracle.OracleTree, count: int, max_len: int = 10**9) -> list[int]:
    """Up to ``count`` leaf nodes (no child node), shortest first: their keys
    are seen only by their own queries, so a node-restricted oracle gives
    their exact dK/dV rows."""
    has_child = np.zeros(len(tree.node_start), dtype=bool)
    has_child[tree.node_parent[tree.node_parent >= 0]] = True
    leaves = [int(n) for n in np.nonzero(~has_child)[0]]
    leaves.sort(key=lambda n: int(tree.node_end[n] - tree.node_start[n]))
    return [n for n in leaves if tree.node_end[n] - tree.node_start[n] + 1 <= max_len][:count]


def node_rows(tree: oracle.OracleTree, nodes: list[int]) -> torch.Tensor:
    return torch.cat([torch.arange(int(tree.node_start[n]), int(tree.node_end[n]) + 1) for n in nodes])


def scale_for(d: int) -> float:
    return 1.0 / math.sqrt(d)
