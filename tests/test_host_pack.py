"""Host-side tests of libtpa (CPU only): the C ABI loads and exports every
symbol include/tpa.h declares, and the native trie packer matches the oracle
bit-exactly on random inputs and on the workloads' sequences."""
import os
import re

import numpy as np
import pytest

import oracle
from oracle.mask import ancestor_pairs
from oracle.pack import PackError
from synth import CONFIGS, make_sequences, random_small_sequences

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def tpa():
    import prefix_shared_tree_attention_gb300 as tpa
    tpa.lib()  # builds the library if needed
    return tpa


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "tpa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tpa_[a-z0-9_]+)\s*\(", src)))


def test_abi_exports_every_declared_symbol(tpa):
    from prefix_shared_tree_attention_gb300._abi import PROTOTYPES
    names = _declared_functions()
    assert len(names) >= 17
    L = tpa.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(PROTOTYPES)
    assert L.tpa_version() >= 100
    assert L.tpa_status_string(0) == b"TPA_OK"
    assert L.tpa_status_string(-3) == b"TPA_ERR_SEQ_TOO_LONG"


def _compare(seqs, mb, tpa):
    pk = oracle.tree_pack(seqs, mb)
    tree = tpa.tree_pack(seqs, mb)
    info = tree.info
    assert info.n_trees == pk.n_trees
    assert info.t_pad == mb
    assert info.total_seq_tokens == pk.total_seq_tokens
    assert info.total_tree_tokens == pk.total_tree_tokens
    assert info.tree_token_ratio == pytest.approx(pk.tree_token_ratio, rel=0, abs=1e-15)
    assert info.ancestor_pairs == sum(ancestor_pairs(t) for t in pk.trees)
    assert info.max_token == max(max(s) for s in seqs)
    assert tree.host_view().max_token == info.max_token
    assert tree.host_view().ancestor_pairs == info.ancestor_pairs
    a = tree.arrays()
    for b, t in enumerate(pk.trees):
        n = t.n
        assert a["n_tokens"][b] == n
        for key in ("tokens", "subtree_end", "parent", "depth", "node_id"):
            got = a[key][b]
            assert np.array_equal(got[:n], getattr(t, key)), (b, key)
            pad = 0 if key == "depth" else -1
            assert np.all(got[n:] == pad), (b, key)
        N = len(t.node_start)
        assert a["n_nodes"][b] == N
        ni = a["node_info"][b]
        assert np.array_equal(ni[:N, 0], t.node_start)
        assert np.array_equal(ni[:N, 1], t.node_end)
        assert np.array_equal(ni[:N, 2], t.node_parent)
        assert np.array_equal(ni[:N, 3], t.node_subtree_end)
        assert np.all(ni[N:] == -1)
        co, cp = a["child_off"][b], a["child_pos"][b]
        assert co[0] == 0 and np.all(co[n:] == co[n])
        for p in range(n):
            assert cp[co[p]:co[p + 1]].tolist() == t.children_of(p)
        assert a["tok_base"][b + 1] - a["tok_base"][b] == n
    assert np.array_equal(a["seq_tree"], pk.seq_tree)
    assert np.array_equal(a["seq_pos"], np.concatenate(pk.seq_pos))
    assert a["seq_off"][0] == 0 and a["seq_off"][-1] == pk.total_seq_tokens


@pytest.mark.parametrize("seed", range(30))
def test_pack_bit_exact_random(tpa, seed):
    rng = np.random.default_rng(1000 + seed)
    seqs = random_small_sequences(rng, int(rng.integers(1, 12)), int(rng.integers(2, 60)),
                                  int(rng.integers(2, 6)))
    mb = 128 * int(rng.integers(1, 4))
    _compare(seqs, mb, tpa)


@pytest.mark.parametrize("seed", range(5))
def test_pack_bit_exact_many_trees(tpa, seed):
    rng = np.random.default_rng(2000 + seed)
    seqs = random_small_sequences(rng, 40, 128, 3, min_len=60)
    _compare(seqs, 256, tpa)


@pytest.mark.parametrize("cid", [1, 2, 3, 5])
def test_pack_bit_exact_workloads(tpa, cid):
    _compare(make_sequences(cid), CONFIGS[cid].max_tokens_per_mb, tpa)


def test_pack_full_tree_takes_only_paths_it_holds(tpa):
    # A tree filled to exactly T_pad still takes a sequence that is a path
    # already in it (no new tokens) and refuses one that adds a single token;
    # a short prefix of its first sequence goes back into it too.
    A = list(range(1, 129))
    seqs = [A, list(A), A[:127] + [999], A[:64], [5] * 64 + [6] * 64]
    _compare(seqs, 128, tpa)
    tree = tpa.tree_pack(seqs, 128)
    assert tree.arrays()["seq_tree"].tolist() == [0, 0, 1, 0, 2]
    assert tree.arrays()["n_tokens"].tolist() == [128, 128, 128]


def test_pack_worked_example(tpa):
    tree = tpa.tree_pack([[0, 1, 2, 3], [0, 1, 4, 5], [0, 6, 7]], 128)
    assert tree.info.total_tree_tokens == 8 and tree.info.total_seq_tokens == 11
    a = tree.arrays()
    assert a["subtree_end"][0, :8].tolist() == [7, 5, 3, 3, 5, 5, 7, 7]


@pytest.mark.parametrize("seqs,mb,code", [
    ([[1, 2]], 100, "TPA_ERR_INVALID_ARG"),
    ([[1, 2]], 0, "TPA_ERR_INVALID_ARG"),
    ([[1], []], 128, "TPA_ERR_EMPTY_SEQUENCE"),
    ([[1] * 129], 128, "TPA_ERR_SEQ_TOO_LONG"),
    ([[1, -5]], 128, "TPA_ERR_INVALID_ARG"),
])
def test_pack_errors(tpa, seqs, mb, code):
    with pytest.raises(tpa.TpaError) as e:
        tpa.tree_pack(seqs, mb)
    assert e.value.name == code
    with pytest.raises(PackError):
        oracle.tree_pack(seqs, mb)


def test_pack_null_and_bad_offsets(tpa):
    import ctypes as C
    L = tpa.lib()
    h = C.c_void_p()
    assert L.tpa_tree_pack(None, None, 1, 128, C.byref(h)) == -1
    toks = (C.c_int32 * 3)(1, 2, 3)
    offs = (C.c_int64 * 2)(1, 3)  # must start at 0
    assert L.tpa_tree_pack(toks, offs, 1, 128, C.byref(h)) == -1
    offs = (C.c_int64 * 3)(0, 2, 1)  # decreasing
    assert L.tpa_tree_pack(toks, offs, 2, 128, C.byref(h)) == -1
    assert L.tpa_tree_get_info(None, None) == -1
    L.tpa_tree_free(None)


def test_blockmask_layout(tpa):
    L = tpa.lib()
    assert L.tpa_blockmask_bytes(0, 128) == 0
    assert L.tpa_blockmask_bytes(1, 100) == 0
    assert L.tpa_blockmask_bytes(2, 1024) > 2 * 8 * 8
    # fp32 gradients: D [B, Hq, T] fp32 only
    assert L.tpa_tree_attn_bwd_workspace_bytes(1, 128, 4, 2, 64, 0) == 4 * 128 * 4
    # bf16 gradients: + fp32 staging dK, dV [B, T, Hkv, d] + counters [B, Hkv, T/128, 16]
    ws = L.tpa_tree_attn_bwd_workspace_bytes(2, 256, 4, 2, 64, 1)
    assert ws >= 2 * 4 * 256 * 4 + 2 * (2 * 256 * 2 * 64 * 4) + 2 * 2 * 2 * 16 * 4
    assert ws < 2 * 4 * 256 * 4 + 2 * (2 * 256 * 2 * 64 * 4) + 2 * 2 * 2 * 16 * 4 + 4 * 256
    assert L.tpa_tree_attn_bwd_workspace_bytes(1, 128, 4, 2, 64, 7) == 0
    assert L.tpa_tree_attn_bwd_workspace_bytes(1, 128, 4, 0, 64, 0) == 0


def test_logprob_calls_refuse_labels_past_vocab(tpa):
    # A tree holding token id 999 cannot be scored against logits rows of
    # 999 or fewer entries: both log-prob entry points refuse the call before
    # any launch (the pointers below are never dereferenced).
    import ctypes as C
    tree = tpa.tree_pack([[1, 2, 999], [1, 5]], 128)
    assert tree.info.max_token == 999
    view = tree.host_view()
    L = tpa.lib()
    fake = 1 << 20
    for vocab in (999, 500, 1):
        assert L.tpa_tree_logprobs_entropy(C.byref(view), fake, 1024, 0, vocab, fake, fake, fake, fake,
                                           None) == -1
        assert L.tpa_lm_head_logprobs_entropy(C.byref(view), fake, fake, 64, vocab, fake, 1 << 40, fake, fake,
                                              fake, fake, None) == -1
