"""GPU parity of the dense ancestor-mask export (tpa_dense_mask; tree
training page, §Megatron 引擎 dense attention-mask tensor) against the
oracle's parent-walk mask, bit-exactly, in both layouts and polarities."""
import numpy as np
import pytest
import torch

import oracle
from oracle.mask import _mask_rows, dense_mask
from synth import random_small_sequences
from _pipeline import check_guards, guarded, pack_and_upload, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tpa():
    import prefix_shared_tree_attention_gb300 as tpa
    tpa.lib()
    tpa.device_check()
    return tpa


def _bits_to_bool(words: np.ndarray) -> np.ndarray:
    w = words.astype(np.int64) & 0xFFFFFFFF
    bits = (w[..., None] >> np.arange(32)) & 1
    return bits.reshape(*words.shape[:-1], -1).astype(bool)


def _check_all(tpa, seqs, mb):
    pk = oracle.tree_pack(seqs, mb)
    tree, dtree, _ = pack_and_upload(tpa, seqs, mb)
    B = tree.n_trees
    got = {}
    for fmt, shape, dt in (("u8", (B, mb, mb), torch.uint8), ("bits", (B, mb, mb // 32), torch.int32)):
        for inv in (False, True):
            buf, view = guarded(shape, dt)           # inside canary guard bands
            tpa.dense_mask(dtree, fmt, invert=inv, out=view)
            torch.cuda.synchronize()
            check_guards(buf, f"{fmt} invert={inv}")
            got[fmt, inv] = view.cpu().numpy()
    u8, u8i = got["u8", False], got["u8", True]
    bits, bitsi = _bits_to_bool(got["bits", False]), _bits_to_bool(got["bits", True])
    for b, t in enumerate(pk.trees):
        ref = dense_mask(t, mb)
        assert np.array_equal(u8[b], ref.astype(np.uint8)), f"tree {b}: u8"
        assert np.array_equal(u8i[b], (~ref).astype(np.uint8)), f"tree {b}: u8 inverted"
        assert np.array_equal(bits[b], ref), f"tree {b}: bits"
        assert np.array_equal(bitsi[b], ~ref), f"tree {b}: bits inverted"


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_dense_mask_random_trees(tpa, seed):
    seqs = random_small_sequences(np.random.default_rng(seed), 24, 90, 3)
    _check_all(tpa, seqs, 256)


def test_dense_mask_config1_full(tpa):
    cfg, seqs = workload(1)
    _check_all(tpa, seqs, cfg.max_tokens_per_mb)


def test_dense_mask_workload_sampled_rows(tpa):
    cfg, seqs = workload(2)
    T = cfg.max_tokens_per_mb
    pk = oracle.tree_pack(seqs, T)
    tree, dtree, _ = pack_and_upload(tpa, seqs, T)
    u8 = tpa.dense_mask(dtree, "u8")
    bits = tpa.dense_mask(dtree, "bits")
    rng = np.random.default_rng(0)
    for b, t in enumerate(pk.trees):
        for r0 in sorted(set(int(x) // 128 * 128 for x in rng.integers(0, T, 3))):
            ref = _mask_rows(t, r0, r0 + 128, T)
            assert np.array_equal(u8[b, r0:r0 + 128].cpu().numpy(), ref.astype(np.uint8)), (b, r0)
            assert np.array_equal(_bits_to_bool(bits[b, r0:r0 + 128].cpu().numpy()), ref), (b, r0)


def test_dense_mask_errors(tpa):
    seqs = random_small_sequences(np.random.default_rng(0), 4, 20, 3)
    tree, dtree, _ = pack_and_upload(tpa, seqs, 128)
    small = torch.empty(10, dtype=torch.uint8, device="cuda")
    with pytest.raises(tpa.TpaError) as e:
        tpa.dense_mask(dtree, "u8", out=small)
    assert e.value.name == "TPA_ERR_BUFFER_TOO_SMALL"
    with pytest.raises(ValueError):
        tpa.dense_mask(dtree, "f32")
    L = tpa.lib()
    assert L.tpa_dense_mask_bytes(2, 256, 0) == 2 * 256 * 256
    assert L.tpa_dense_mask_bytes(2, 256, 1) == 2 * 256 * 256 // 8
    assert L.tpa_dense_mask_bytes(2, 100, 0) == 0
