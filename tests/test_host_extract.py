"""Host-side parity of sequence extraction and padded packing
(tpa_extract_sequences, tpa_tree_pack_padded; tree training page, §树构建过程
step 1) against the oracle, bit-exactly."""
import numpy as np
import pytest

import oracle
from oracle.extract import extract_sequences
from synth import CONFIGS, make_sequences


def _blob(tpa, tree):
    import ctypes
    return ctypes.string_at(tpa.lib().tpa_tree_host_blob(tree._h), tree.info.blob_bytes)


@pytest.fixture(scope="session")
def tpa():
    import prefix_shared_tree_attention_gb300 as tpa
    tpa.lib()
    return tpa


def _padded_batch(seqs, rng, side):
    L = max(len(s) for s in seqs) + int(rng.integers(0, 5))
    ids = rng.integers(0, 50, size=(len(seqs), L)).astype(np.int32)  # junk in the padding
    mask = np.zeros((len(seqs), L), dtype=np.uint8)
    for r, s in enumerate(seqs):
        if side == "right":
            cols = np.arange(len(s))
        elif side == "left":
            cols = np.arange(L - len(s), L)
        else:  # interior gaps
            cols = np.sort(rng.choice(L, size=len(s), replace=False))
        ids[r, cols] = s
        mask[r, cols] = 1
    return ids, mask


@pytest.mark.parametrize("side", ["right", "left", "gaps"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_extract_bit_exact(tpa, side, seed):
    rng = np.random.default_rng(seed)
    seqs = [rng.integers(0, 6, size=int(rng.integers(1, 40))).tolist() for _ in range(int(rng.integers(1, 30)))]
    ids, mask = _padded_batch(seqs, rng, side)
    want = extract_sequences(ids, mask)
    assert want == seqs
    toks, offs = tpa.extract_sequences(ids, mask)
    got = [toks[offs[r]:offs[r + 1]].tolist() for r in range(len(seqs))]
    assert got == want


@pytest.mark.parametrize("cid", [1, 2])
def test_pack_padded_matches_oracle(tpa, cid):
    rng = np.random.default_rng(cid)
    seqs = make_sequences(cid)
    ids, mask = _padded_batch(seqs, rng, "left")
    mb = CONFIGS[cid].max_tokens_per_mb
    t = tpa.tree_pack_padded(ids, mask, mb)
    pk = oracle.tree_pack(extract_sequences(ids, mask), mb)
    assert t.n_trees == pk.n_trees
    assert t.info.total_tree_tokens == pk.total_tree_tokens
    ref = tpa.tree_pack(seqs, mb)
    assert _blob(tpa, t) == _blob(tpa, ref)  # identical packing, byte for byte


def test_empty_row_is_rejected(tpa):
    ids = np.array([[1, 2], [3, 4]], dtype=np.int32)
    mask = np.array([[1, 1], [0, 0]], dtype=np.uint8)
    toks, offs = tpa.extract_sequences(ids, mask)
    assert offs.tolist() == [0, 2, 2]
    with pytest.raises(tpa.TpaError) as e:
        tpa.tree_pack_padded(ids, mask, 128)
    assert e.value.name == "TPA_ERR_EMPTY_SEQUENCE"
    with pytest.raises(ValueError):
        tpa.extract_sequences(ids, mask[:1])
