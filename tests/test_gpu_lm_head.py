"""GPU parity of the fused LM-head log-prob pass (tpa_lm_head_logprobs_entropy)
against the oracle: fp64 logits = hidden @ weight^T fed to the §对数概率计算
definition; log-probs and entropies within 1e-3 absolute."""
import numpy as np
import pytest
import torch

import oracle
from oracle.lm_head import LazyLogits
from oracle.logprobs import position_logprobs_entropy, sequence_logprobs_entropy
from synth import make_hidden, make_lm_weight, random_small_sequences
from _pipeline import LOGP_ABS, pack_and_upload, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tpa():
    import prefix_shared_tree_attention_gb300 as tpa
    tpa.lib()
    tpa.device_check()
    return tpa


def _run(tpa, seqs, mb, V, H, cid):
    pk = oracle.tree_pack(seqs, mb)
    tree, dtree, _ = pack_and_upload(tpa, seqs, mb)
    rows = tree.info.total_tree_tokens
    hid = make_hidden(cid, rows, H, "cuda")
    w = make_lm_weight(cid, V, H, "cuda")
    out = tpa.lm_head_logprobs_entropy(dtree, hid, w)
    tpa.sync_status()
    return pk, tree, hid.cpu(), w.cpu(), [x.cpu() for x in out]


def _row_base(pk):
    base, acc = [], 0
    for t in pk.trees:
        base.append(acc)
        acc += t.n
    return base


def _check_full(pk, seqs, hid, w, out):
    pl, pe, sl, se = out
    lg = LazyLogits(hid, w)
    rb = _row_base(pk)
    lp, ent = sequence_logprobs_entropy(pk, seqs, lg, rb)
    got_lp = sl.numpy().astype(np.float64)
    got_ent = se.numpy().astype(np.float64)
    off = 0
    for s in range(len(seqs)):
        L = len(seqs[s])
        assert np.abs(got_lp[off:off + L] - lp[s]).max() <= LOGP_ABS, f"seq {s} logp"
        assert np.abs(got_ent[off:off + L] - ent[s]).max() <= LOGP_ABS, f"seq {s} entropy"
        off += L
    for b, t in enumerate(pk.trees):
        plp, pen = position_logprobs_entropy(pk, lg, rb, b)
        assert np.abs(pl[b, :t.n].numpy() - plp).max() <= LOGP_ABS, f"tree {b} pos_logp"
        assert np.abs(pe[b, :t.n].numpy() - pen).max() <= LOGP_ABS, f"tree {b} pos_entropy"
        assert (pl[b, t.n:] == 0).all() and (pe[b, t.n:] == 0).all(), f"tree {b} padding"


@pytest.mark.parametrize("V,H", [(1000, 256), (257, 64), (200, 128), (2304, 192)])
def test_lm_head_small_full(tpa, V, H):
    # several trees, ragged row tiles, vocab tails (1000 % 256, 257, one partial tile)
    seqs = random_small_sequences(np.random.default_rng(V), 24, 90, min(V, 50))
    pk, tree, hid, w, out = _run(tpa, seqs, 256, V, H, 1)
    assert pk.n_trees > 1
    _check_full(pk, seqs, hid, w, out)


def test_lm_head_tiny_tree(tpa):
    # fewer rows than one CTA's 128: the pair's second CTA has no real row and
    # its hidden-row loads lie wholly past the end (zero fill)
    seqs = random_small_sequences(np.random.default_rng(77), 4, 20, 30)
    pk, tree, hid, w, out = _run(tpa, seqs, 128, 300, 64, 2)
    assert tree.info.total_tree_tokens < 128
    _check_full(pk, seqs, hid, w, out)


def test_lm_head_config1_full(tpa):
    cfg, seqs = workload(1)
    pk, tree, hid, w, out = _run(tpa, seqs, cfg.max_tokens_per_mb, 1000, 512, 1)
    _check_full(pk, seqs, hid, w, out)


@pytest.mark.parametrize("H", [1024, 4096])
def test_lm_head_qwen_vocab_sampled(tpa, H):
    # the logits workload's vocabulary on the GRPO-shaped trees: sampled
    # positions of every tree, and every position of the two shortest
    # sequences; H 4096 is the hidden size bench.py times
    cfg, seqs = workload(2)
    V = 151936
    pk, tree, hid, w, out = _run(tpa, seqs, cfg.max_tokens_per_mb, V, H, 4)
    pl, pe, sl, se = out
    lg = LazyLogits(hid, w)
    rb = _row_base(pk)
    rng = np.random.default_rng(4)
    for b in range(pk.n_trees):
        t = pk.trees[b]
        pos = sorted(set(int(x) for x in rng.integers(0, t.n, 3)))
        plp, pen = position_logprobs_entropy(pk, lg, rb, b, pos)
        assert np.abs(pl[b, pos].numpy() - plp).max() <= LOGP_ABS, f"tree {b} pos_logp"
        assert np.abs(pe[b, pos].numpy() - pen).max() <= LOGP_ABS, f"tree {b} pos_entropy"
        assert (pl[b, t.n:] == 0).all() and (pe[b, t.n:] == 0).all()
    shortest = sorted(range(len(seqs)), key=lambda s_: len(seqs[s_]))[:2]
    lp, ent = sequence_logprobs_entropy(pk, seqs, lg, rb, shortest)
    offs = np.concatenate([[0], np.cumsum([len(s_) for s_ in seqs])])
    for u, s_ in enumerate(shortest):
        got_lp = sl[offs[s_]:offs[s_ + 1]].numpy().astype(np.float64)
        got_ent = se[offs[s_]:offs[s_ + 1]].numpy().astype(np.float64)
        assert np.abs(got_lp - lp[u]).max() <= LOGP_ABS, f"seq {s_} logp"
        assert np.abs(got_ent - ent[u]).max() <= LOGP_ABS, f"seq {s_} entropy"
    assert torch.isfinite(sl).all() and torch.isfinite(se).all()


def test_lm_head_errors(tpa):
    seqs = random_small_sequences(np.random.default_rng(0), 4, 20, 3)
    tree, dtree, _ = pack_and_upload(tpa, seqs, 128)
    rows = tree.info.total_tree_tokens
    hid = torch.zeros((rows, 96), dtype=torch.bfloat16, device="cuda")  # H not a multiple of 64
    w = torch.zeros((10, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tpa.TpaError) as e:
        tpa.lm_head_logprobs_entropy(dtree, hid, w)
    assert e.value.name == "TPA_ERR_INVALID_ARG"
    hid = torch.zeros((rows, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((10, 64), dtype=torch.bfloat16, device="cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(tpa.TpaError) as e:
        tpa.lm_head_logprobs_entropy(dtree, hid, w, workspace=small)
    assert e.value.name == "TPA_ERR_BUFFER_TOO_SMALL"
    with pytest.raises(ValueError):
        tpa.lm_head_logprobs_entropy(dtree, hid[:-1], w)
