"""Maximum sizes (GPU): max_tokens_per_mb = 131072, the packer's limit (1024
blocks a side).

* A small tree padded to 131072 positions: block classes and both CSR lists
  bit-exact against the oracle, every output of the forward and backward
  against the oracle, and the padding rows zero.
* One 131072-token sequence (a single chain, 8.6e9 ancestor pairs): the block
  classes against the closed form of a causal chain (FULL below the
  diagonal, PARTIAL on it, EMPTY above), and sampled rows of O, LSE and dQ,
  plus dK/dV of the last key tile (seen only by the last tile's queries),
  against the oracle computed one query row at a time.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.mask import block_classes, block_csr
from synth import random_small_sequences
from _pipeline import assert_attn_close, assert_attn_close_bf16_out, pack_and_upload, random_inputs

pytestmark = pytest.mark.gpu

T_MAX = 131072


@pytest.fixture(scope="module")
def tpa():
    import prefix_shared_tree_attention_gb300 as tpa
    tpa.lib()
    tpa.device_check()
    return tpa


def test_small_tree_in_maximum_padding(tpa):
    rng = np.random.default_rng(131)
    seqs = random_small_sequences(rng, 12, 400, 3, min_len=1)
    pk = oracle.tree_pack(seqs, T_MAX)
    tree, dtree, mask = pack_and_upload(tpa, seqs, T_MAX)
    t = pk.trees[0]
    arr = mask.arrays()
    cls = block_classes(t, T_MAX)
    assert np.array_equal(arr["cls"][0].cpu().numpy(), cls)
    csr = block_csr(cls)
    nq = len(csr["q_idx"])
    for key in ("q_ptr", "k_ptr"):
        assert np.array_equal(arr[key][0].cpu().numpy(), csr[key])
    for key in ("q_idx", "k_idx"):
        assert np.array_equal(arr[key][0][:nq].cpu().numpy(), csr[key])
    (q, k, v, do), (qc, kc, vc, doc) = random_inputs(1, T_MAX, 2, 1, 64, 13)
    o, lse = tpa.tree_attn_fwd(dtree, mask, q, k, v)
    dq, dk, dv = tpa.tree_attn_bwd(dtree, mask, q, k, v, o, lse, do)
    tpa.sync_status()
    n = t.n
    O, L = oracle.attn_forward(t, qc[0, :n], kc[0, :n], vc[0, :n])
    dQ, dK, dV = oracle.attn_backward(t, qc[0, :n], kc[0, :n], vc[0, :n], doc[0, :n])
    assert_attn_close(o[0, :n], O, "O")
    assert_attn_close(lse[0, :, :n], L, "LSE", max_abs=2e-3, rel_l2=1e-4)
    for name, g, r in (("dQ", dq, dQ), ("dK", dk, dK), ("dV", dv, dV)):
        assert_attn_close(g[0, :n], r, name)
        assert torch.all(g[0, n:] == 0), f"{name} padding"
    assert torch.all(o[0, n:] == 0) and torch.all(lse[0, :, n:] == 0)


def test_one_chain_of_maximum_length(tpa):
    rng = np.random.default_rng(132)
    seq = rng.integers(0, 32000, size=T_MAX).tolist()
    pk = oracle.tree_pack([seq], T_MAX)
    t = pk.trees[0]
    assert pk.n_trees == 1 and t.n == T_MAX and len(t.node_start) == 1
    tree, dtree, mask = pack_and_upload(tpa, [seq], T_MAX)
    nb = T_MAX // 128
    cls = mask.arrays()["cls"][0].cpu().numpy()
    qb, kb = np.meshgrid(np.arange(nb), np.arange(nb), indexing="ij")
    expect = np.where(kb < qb, 2, np.where(kb == qb, 1, 0)).astype(np.uint8)  # FULL / PARTIAL / EMPTY
    assert np.array_equal(cls, expect)
    arr = mask.arrays()
    assert np.array_equal(arr["q_ptr"][0].cpu().numpy(), np.cumsum(np.r_[0, np.arange(1, nb + 1)]))
    hq, hkv, d = 2, 1, 64
    (q, k, v, do), (qc, kc, vc, doc) = random_inputs(1, T_MAX, hq, hkv, d, 17)
    o, lse = tpa.tree_attn_fwd(dtree, mask, q, k, v)
    grads = {gdt: tpa.tree_attn_bwd(dtree, mask, q, k, v, o, lse, do, grad_dtype=gdt)
             for gdt in (torch.float32, torch.bfloat16)}
    tpa.sync_status()
    last = list(range(T_MAX - 128, T_MAX))   # every query that sees the last key tile
    sample = sorted({0, 1, 127, 128, 4095, 65535, 65536} | set(rng.integers(0, T_MAX - 128, 6).tolist()))
    rows = sample + last
    O, L, dQ, dK, dV = oracle.attn_rows(t, qc[0], kc[0], vc[0], rows, dO=doc[0])
    idx = torch.as_tensor(rows)
    assert_attn_close(o[0].cpu()[idx], O, "O sampled rows")
    assert_attn_close(lse[0].cpu()[:, idx], L, "LSE sampled rows", max_abs=2e-3, rel_l2=1e-4)
    dK_last, dV_last = dK[T_MAX - 128:], dV[T_MAX - 128:]
    for gdt, close in ((torch.float32, assert_attn_close), (torch.bfloat16, assert_attn_close_bf16_out)):
        dq, dk, dv = grads[gdt]
        close(dq[0].cpu()[idx], dQ, f"{gdt} dQ sampled rows")
        close(dk[0, T_MAX - 128:].cpu(), dK_last, f"{gdt} dK last key tile")
        close(dv[0, T_MAX - 128:].cpu(), dV_last, f"{gdt} dV last key tile")
