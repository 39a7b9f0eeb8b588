"""Host-side parity of the native micro-batch / rank balancing (tpa_balance,
tpa_packing_metrics) against the oracle (blog post "AReaL 序列打包算法 FFD 与
KK"): group assignments must match bit-exactly, metrics to rounding."""
import random

import numpy as np
import pytest

from oracle.balance import BalanceError, ffd_allocate, group_of, kk_allocate, packing_metrics
from synth import CONFIGS, make_sequences

CODES = {"INVALID_ARG": "TPA_ERR_INVALID_ARG", "SEQ_TOO_LONG": "TPA_ERR_SEQ_TOO_LONG"}


@pytest.fixture(scope="session")
def tpa():
    import prefix_shared_tree_attention_gb300 as tpa
    tpa.lib()
    return tpa


def _instances(seed):
    rng = random.Random(seed)
    out = []
    for _ in range(60):
        kind = rng.choice(["uniform", "bimodal", "ties"])
        n = rng.randint(1, 200)
        if kind == "uniform":
            w = [rng.randint(1, 1000) for _ in range(n)]
        elif kind == "bimodal":
            w = [rng.randint(800, 2048) if rng.random() < 0.3 else rng.randint(50, 200) for _ in range(n)]
        else:
            w = [rng.choice([64, 128, 256]) for _ in range(n)]
        cap = rng.choice([max(w), max(w) * 2, max(w) * 5, 10**12])
        mg = rng.randint(1, max(1, min(n, 8)))
        div = rng.choice([1, 1, 2, 4])
        out.append((w, cap, mg, div))
    return out


def _native(tpa, w, cap, mg, div, algo):
    try:
        g, ng, used = tpa.balance(w, cap, mg, div, algo)
        return list(map(int, g)), ng, used, None
    except tpa.TpaError as e:
        return None, None, None, e.name


def _oracle(w, cap, mg, div, algo):
    try:
        if algo == "ffd":
            groups, used = ffd_allocate(w, cap, mg, div), "ffd"
        else:
            groups, used = kk_allocate(w, cap, mg, div)
        return group_of(groups, len(w)), len(groups), used, None
    except BalanceError as e:
        return None, None, None, CODES[e.code]


@pytest.mark.parametrize("algo", ["ffd", "kk"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_balance_bit_exact(tpa, algo, seed):
    for w, cap, mg, div in _instances(seed * 10 + (algo == "kk")):
        assert _native(tpa, w, cap, mg, div, algo) == _oracle(w, cap, mg, div, algo), (w, cap, mg, div)


def test_balance_hand_cases(tpa):
    g, ng, used = tpa.balance([5, 4, 3, 2, 1], 6)
    assert list(g) == [0, 1, 2, 2, 1] and ng == 3 and used == "ffd"
    g, ng, used = tpa.balance([3, 3, 2, 2, 2], 6, algorithm="kk")
    assert used == "ffd" and list(g) == [0, 0, 1, 1, 1]


def test_balance_trees_of_the_workloads(tpa):
    # trees -> ranks by tree tokens, and sequences -> micro-batches by length
    for cid in (2, 3, 5):
        seqs = make_sequences(cid)
        lens = [len(s) for s in seqs]
        cap = CONFIGS[cid].max_tokens_per_mb
        for algo in ("ffd", "kk"):
            assert _native(tpa, lens, cap, 2, 1, algo) == _oracle(lens, cap, 2, 1, algo)
            assert _native(tpa, lens, 10**12, 4, 1, algo) == _oracle(lens, 10**12, 4, 1, algo)


def test_metrics_match_oracle(tpa):
    rng = random.Random(7)
    for _ in range(40):
        n = rng.randint(1, 100)
        w = [rng.randint(1, 500) for _ in range(n)]
        ng = rng.randint(1, n)
        g = [rng.randrange(ng) for _ in range(n)]
        cap = rng.randint(500, 5000)
        m = tpa.packing_metrics(w, g, ng, cap)
        groups = [[i for i in range(n) if g[i] == k] for k in range(ng)]
        o = packing_metrics(w, groups, cap)
        for f in ("n_groups", "total", "max_load", "min_load", "spread", "wasted"):
            assert m[f] == getattr(o, f), f
        for f in ("mean", "std_dev", "cv", "imbalance_ratio", "utilization"):
            assert m[f] == pytest.approx(getattr(o, f), rel=1e-12, abs=1e-12), f


@pytest.mark.parametrize("w,cap,mg,div,code", [
    ([5, 7], 6, 1, 1, "TPA_ERR_SEQ_TOO_LONG"),
    ([1, 0], 10, 1, 1, "TPA_ERR_INVALID_ARG"),
    ([1, 2], 10, 3, 1, "TPA_ERR_INVALID_ARG"),
    ([1, 2, 3], 10, 1, 0, "TPA_ERR_INVALID_ARG"),
    ([1, 2, 3], 0, 1, 1, "TPA_ERR_INVALID_ARG"),
])
def test_balance_errors(tpa, w, cap, mg, div, code):
    for algo in ("ffd", "kk"):
        assert _native(tpa, w, cap, mg, div, algo)[3] == code
    with pytest.raises(ValueError):
        tpa.balance([1, 2], 10, algorithm="best")
    with pytest.raises(tpa.TpaError):
        tpa.packing_metrics([1, 2], [0, 2], 2, 10)
