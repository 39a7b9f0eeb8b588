"""Pins for the oracle FFD / KK balancing and packing metrics (blog post
"AReaL 序列打包算法 FFD 与 KK": FFD puts each item, heaviest first, into the
lightest group that fits; KK is the k-way largest differencing method; the
post's test asserts that KK balances no worse than FFD)."""
import heapq
import itertools
import random

import pytest

from oracle.balance import BalanceError, ffd_allocate, group_of, kk_allocate, packing_metrics


def loads(weights, groups):
    return [sum(weights[i] for i in g) for g in groups]


def test_ffd_lightest_fit_hand_case():
    # weights 5,4,3,2,1 with capacity 6: 5 -> new, 4 -> new, 3 -> new (no room),
    # 2 -> the lightest that fits is the 3 (not the 4, which first fit would take),
    # 1 -> the lightest that fits is now the 4.
    w = [5, 4, 3, 2, 1]
    groups = ffd_allocate(w, 6)
    assert groups == [[0], [1, 4], [2, 3]]
    assert loads(w, groups) == [5, 5, 5]


def test_ffd_min_groups_and_divisor_retry():
    # min_groups 3 gives 3 groups; the divisor 2 forces a retry with 4.
    w = [1, 1, 1, 1, 1]
    assert len(ffd_allocate(w, 100, min_groups=3)) == 3
    groups = ffd_allocate(w, 100, min_groups=3, divisor=2)
    assert groups == [[0, 4], [1], [2], [3]]


def test_ffd_respects_capacity_and_covers_items():
    rng = random.Random(3)
    for _ in range(50):
        w = [rng.randint(1, 50) for _ in range(rng.randint(1, 40))]
        cap = rng.randint(50, 120)
        groups = ffd_allocate(w, cap, min_groups=rng.randint(1, 3) if len(w) >= 3 else 1)
        assert sorted(itertools.chain(*groups)) == list(range(len(w)))
        assert max(loads(w, groups)) <= cap


def test_kk_two_way_spread_is_the_differencing_value():
    # Two-way KK: merging two states leaves |spread_a - spread_b|, so the final
    # spread is the classic Karmarkar-Karp differencing of the numbers.
    rng = random.Random(5)
    for _ in range(40):
        w = [rng.randint(1, 1000) for _ in range(rng.randint(2, 30))]
        h = [-x for x in w]
        heapq.heapify(h)
        while len(h) > 1:
            a, b = -heapq.heappop(h), -heapq.heappop(h)
            heapq.heappush(h, -(a - b))
        groups, algo = kk_allocate(w, 10**12, min_groups=2)
        assert algo == "kk" and len(groups) == 2
        ld = loads(w, groups)
        assert max(ld) - min(ld) == -h[0]


def test_kk_partition_and_singletons():
    w = [7, 3, 9, 1]
    groups, algo = kk_allocate(w, 10**12, min_groups=4)
    assert algo == "kk" and sorted(map(tuple, groups)) == [(0,), (1,), (2,), (3,)]
    assert loads(w, groups) == [9, 7, 3, 1]  # numbered heaviest first
    rng = random.Random(9)
    for _ in range(30):
        w = [rng.randint(1, 100) for _ in range(rng.randint(3, 25))]
        groups, _ = kk_allocate(w, 10**12, min_groups=3)
        assert sorted(itertools.chain(*groups)) == list(range(len(w)))


def test_kk_group_count_from_capacity_and_divisor():
    w = [10] * 10  # total 100, capacity 30 -> ceil = 4, divisor 3 -> 6 groups
    groups, algo = kk_allocate(w, 30, min_groups=1, divisor=3)
    assert algo == "kk" and len(groups) == 6 and max(loads(w, groups)) <= 30


def test_kk_falls_back_to_ffd_over_capacity():
    # KK (greedy differencing) reaches loads 7 / 5 here; with capacity 6 the
    # result is discarded and FFD's {3,3} / {2,2,2} is returned.
    w = [3, 3, 2, 2, 2]
    groups, algo = kk_allocate(w, 6)
    assert algo == "ffd"
    assert groups == [[0, 1], [2, 3, 4]]


def bimodal(rng, n):
    # the post's simulation: short 50-200, long 800-2048, 30 % long
    return [rng.randint(800, 2048) if rng.random() < 0.3 else rng.randint(50, 200) for _ in range(n)]


def test_kk_balances_no_worse_than_ffd_on_bimodal_lengths():
    rng = random.Random(11)
    wins = trials = 0
    kk_sum = ffd_sum = 0
    for _ in range(40):
        w = bimodal(rng, 64)
        f = ffd_allocate(w, 10**12, min_groups=4)
        k, algo = kk_allocate(w, 10**12, min_groups=4)
        fs = max(loads(w, f)) - min(loads(w, f))
        ks = max(loads(w, k)) - min(loads(w, k))
        trials += 1
        wins += ks <= fs
        kk_sum += ks
        ffd_sum += fs
    assert wins >= 0.9 * trials and kk_sum < ffd_sum


def test_brute_force_tiny():
    rng = random.Random(2)
    for _ in range(60):
        n = rng.randint(2, 7)
        k = rng.randint(2, min(3, n))
        w = [rng.randint(1, 20) for _ in range(n)]
        best = min(max(s) - min(s) for s in (
            [sum(w[i] for i in range(n) if a[i] == g) for g in range(k)]
            for a in itertools.product(range(k), repeat=n)))
        groups, _ = kk_allocate(w, 10**12, min_groups=k)
        ld = loads(w, groups)
        assert max(ld) - min(ld) >= best
        assert max(ld) - min(ld) <= max(w)  # differencing never leaves more than the largest item


def test_metrics_closed_forms():
    w = [2, 4]
    m = packing_metrics(w, [[0], [1]], capacity=5)
    assert (m.spread, m.max_load, m.min_load, m.total) == (2, 4, 2, 6)
    assert m.mean == 3 and m.std_dev == 1 and m.cv == pytest.approx(1 / 3)
    assert m.imbalance_ratio == pytest.approx(4 / 3)
    assert m.utilization == pytest.approx(6 / 10) and m.wasted == 4


def test_errors():
    with pytest.raises(BalanceError):
        ffd_allocate([5, 7], 6)  # heavier than the capacity
    with pytest.raises(BalanceError):
        kk_allocate([1, 2], 100, min_groups=3)  # more groups than items
    with pytest.raises(BalanceError):
        ffd_allocate([1, 0], 100)
    assert group_of([[1], [0, 2]], 3) == [1, 0, 1]
