"""GPU parity of the backward on keys that many queries share (GPU).

On a packed tree the keys of a shared prefix are seen by every query below
them (tree training page, §树构建过程: shared prefixes are computed once), so
their dK/dV rows sum contributions from whole subtrees.  In the KV kernel
such a key tile has a long column of (query head, query tile) steps; a
column longer than one work item is split into several items that add into
rows the preprocess zeroed: the outputs for fp32 gradients, fp32 staging rows
that the last item converts for bf16 gradients.  These tests compare EVERY
dQ, dK and dV row of such trees with the oracle, element by element:

* a mid-size tree with a 3072-token shared prefix and four branches, at d 128
  (CTA-pair dQ kernel) and d 64 (single-CTA dQ kernel), fp32 and bf16
  gradients, called twice with different inputs on the same buffers so that
  rows left over from the first call would show;
* the full-size GRPO-shaped and agentic workloads, on every row of their
  first tree, for one key/value head and the query heads of its group
  (heads are independent, so the oracle run on that slice gives the exact
  values of those heads).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.mask import block_classes
from _pipeline import (assert_attn_close, assert_attn_close_bf16_out, check_guards, guarded, pack_and_upload,
                       random_inputs, workload, workload_tensors)

pytestmark = pytest.mark.gpu


def kv_chunk(pk, hq: int, group: int, t_pad: int) -> int:
    """Steps per KV work item, by the rule tpa.h states: a quarter of one SM's
    share of the estimated steps (ancestor pairs of all trees x Hq / 128^2),
    at least 64, at most a whole column (group x T_pad / 128)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    pairs = sum(int((t.depth[:t.n] + 1).sum()) for t in pk.trees)
    est = pairs * hq // (128 * 128)
    return int(min(max(est // (sms * 4), 64), group * (t_pad // 128)))


@pytest.fixture(scope="module")
def tpa():
    import prefix_shared_tree_attention_gb300 as tpa
    tpa.lib()
    tpa.device_check()
    return tpa


def _longest_column(tree, t_pad: int) -> int:
    """Non-empty query tiles of the most-seen key tile (from the oracle's classes)."""
    cls = block_classes(tree, t_pad)
    return int((cls != 0).sum(axis=0).max())


def _shared_prefix_seqs(prefix_len: int, n_branch: int, branch_len: int, seed: int) -> list[list[int]]:
    rng = np.random.default_rng(seed)
    prefix = rng.integers(0, 32000, size=prefix_len).tolist()
    return [prefix + [40000 + 1000 * b + i for i in range(branch_len)] for b in range(n_branch)]


@pytest.mark.parametrize("hq,hkv,d", [(8, 1, 128), (4, 1, 64), (8, 2, 128)])
def test_shared_prefix_every_row(tpa, hq, hkv, d):
    T = 4096
    seqs = _shared_prefix_seqs(3072, 4, 256, seed=hq * 10 + d)
    pk = oracle.tree_pack(seqs, T)
    assert pk.n_trees == 1 and pk.trees[0].n == T
    # the prefix's first key tile is seen by all 32 query tiles: G * 32 steps,
    # more than one work item, so the split-and-add paths run (fp32 outputs,
    # bf16 staging rows)
    assert (hq // hkv) * _longest_column(pk.trees[0], T) > kv_chunk(pk, hq, hq // hkv, T)
    tree, dtree, mask = pack_and_upload(tpa, seqs, T)
    t = pk.trees[0]
    # outputs start as NaN (rows no item writes would show) inside canary guard bands
    guards = {gdt: [guarded(x, gdt) for x in ((1, T, hq, d), (1, T, hkv, d), (1, T, hkv, d))]
              for gdt in (torch.float32, torch.bfloat16)}
    for gs in guards.values():
        for _, view in gs:
            view.fill_(float("nan"))
    bufs = {gdt: tuple(view for _, view in gs) for gdt, gs in guards.items()}
    for call, seed in enumerate((31, 32)):   # same output buffers, new inputs
        (q, k, v, do), (qc, kc, vc, doc) = random_inputs(1, T, hq, hkv, d, seed)
        o, lse = tpa.tree_attn_fwd(dtree, mask, q, k, v)
        got = {gdt: tpa.tree_attn_bwd(dtree, mask, q, k, v, o, lse, do, grad_dtype=gdt, out=bufs[gdt])
               for gdt in bufs}
        tpa.sync_status()
        for gdt, gs in guards.items():
            for name, (buf, _) in zip(("dQ", "dK", "dV"), gs):
                check_guards(buf, f"{gdt} {name}")
        O, _ = oracle.attn_forward(t, qc[0], kc[0], vc[0], t_pad=T)
        assert_attn_close(o[0], O, f"call {call} O")
        ref = oracle.attn_backward(t, qc[0], kc[0], vc[0], doc[0], t_pad=T)
        for name, g, r in zip(("dQ", "dK", "dV"), got[torch.float32], ref):
            assert_attn_close(g[0], r, f"call {call} fp32 {name}")
        for name, g, r in zip(("dQ", "dK", "dV"), got[torch.bfloat16], ref):
            assert_attn_close_bf16_out(g[0], r, f"call {call} bf16 {name}")
        # the root tile's rows, the ones every query adds into, on their own
        for name, g, r in zip(("dK", "dV"), got[torch.float32][1:], ref[1:]):
            assert_attn_close(g[0, :128], r[:128], f"call {call} fp32 {name} root tile")


@pytest.mark.parametrize("cid", [2, 3])
def test_workload_first_tree_one_kv_group(tpa, cid):
    """Every row of tree 0 of the full-size workload, for kv head 0 and query
    heads 0 .. G-1, fp32 and bf16 gradients."""
    cfg, seqs = workload(cid)
    T = cfg.max_tokens_per_mb
    G = cfg.n_heads_q // cfg.n_heads_kv
    pk = oracle.tree_pack(seqs, T)
    t = pk.trees[0]
    assert G * _longest_column(t, T) > kv_chunk(pk, cfg.n_heads_q, G, T)
    tree, dtree, mask = pack_and_upload(tpa, seqs, T)
    q, k, v, do = workload_tensors(cid, tree.n_trees, T)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = tpa.tree_attn_fwd(dtree, mask, qd, kd, vd)
    f32 = tpa.tree_attn_bwd(dtree, mask, qd, kd, vd, o, lse, dod)
    b16 = tpa.tree_attn_bwd(dtree, mask, qd, kd, vd, o, lse, dod, grad_dtype=torch.bfloat16)
    tpa.sync_status()
    n = t.n
    dQ, dK, dV = oracle.attn_backward(t, q[0, :, :G], k[0, :, :1], v[0, :, :1], do[0, :, :G], t_pad=T)
    for tag, (dq, dk, dv), close in (("fp32", f32, assert_attn_close), ("bf16", b16, assert_attn_close_bf16_out)):
        close(dq[0, :n, :G].cpu(), dQ[:n], f"cfg{cid} {tag} dQ heads 0..{G - 1}")
        close(dk[0, :n, :1].cpu(), dK[:n], f"cfg{cid} {tag} dK kv head 0")
        close(dv[0, :n, :1].cpu(), dV[:n], f"cfg{cid} {tag} dV kv head 0")
        # the root node's rows (the shared prefix) on their own
        r1 = int(t.node_end[0]) + 1
        close(dk[0, :r1, :1].cpu(), dK[:r1], f"cfg{cid} {tag} dK root node")
        close(dv[0, :r1, :1].cpu(), dV[:r1], f"cfg{cid} {tag} dV root node")
        assert torch.all(dk[0, n:] == 0) and torch.all(dv[0, n:] == 0) and torch.all(dq[0, n:] == 0)
