"""Oracle micro-batch / rank balancing (test infrastructure; see the package
docstring).

Follows the blog post "AReaL 序列打包算法 FFD 与 KK" (micro-batch load
balancing), sections on FFD (First Fit Decreasing), KK (Karmarkar-Karp
largest differencing) and the packing metrics.  In tree training the items
are packed trees (or sequences) and a group is a micro-batch or a DP rank.

FFD, as the post describes it:
  * take items by weight, heaviest first;
  * while fewer than ``min_groups`` groups exist, an item opens a new group;
  * otherwise it goes to the LIGHTEST group that can still take it
    (load + weight <= capacity); if none can, it opens a new group;
  * the final group count must be >= ``min_groups`` and a multiple of
    ``groups_divisor``; if it is not, ``min_groups`` is raised to the next
    multiple of the divisor and the whole allocation is redone.

KK (k-way largest differencing, Korf 2009, as the post describes it):
  * k = max(min_groups, ceil(total / capacity)), rounded up to a multiple of
    ``groups_divisor``; it may not exceed the number of items;
  * every item starts as a partial partition ("state") of k sets: the item
    alone in one set, the other k-1 sets empty;
  * a max-heap orders states by spread (largest set sum minus smallest);
    the two states with the largest spread are popped and merged by pairing
    the i-th largest set of the first with the i-th smallest set of the
    second; the merged state is pushed back; this repeats until one state
    remains;
  * if a final set exceeds the capacity the result is discarded and FFD is
    used instead.

Readings (the post leaves these open; each is a fixed rule here):
  * weight ties keep input order (stable); equal group loads go to the
    earliest-created group;
  * heap ties (equal spread) pop the state created first (items are created
    in input order, merged states after them in merge order); within a
    state, equal set sums keep their current set order when sorted;
  * FFD groups are numbered in creation order; KK groups are numbered by the
    final state's sets ordered by sum, heaviest first (ties keep set order);
  * an item heavier than the capacity, a non-positive weight, or a required
    group count above the number of items is an error;
  * metrics: spread = max - min load; imbalance_ratio = max / mean;
    std_dev = population standard deviation of the loads; cv = std_dev /
    mean; utilization = total / (groups * capacity); wasted = groups *
    capacity - total (tokens of padding if every group is filled to the
    capacity).
"""
from __future__ import annotations

import math
from dataclasses import dataclass


class BalanceError(ValueError):
    def __init__(self, code: str, msg: str):
        super().__init__(f"{code}: {msg}")
        self.code = code


def _check(weights, capacity, min_groups, divisor):
    if len(weights) < 1:
        raise BalanceError("INVALID_ARG", "no items")
    if capacity < 1 or min_groups < 1 or divisor < 1:
        raise BalanceError("INVALID_ARG", "capacity, min_groups and divisor must be positive")
    for w in weights:
        if w <= 0:
            raise BalanceError("INVALID_ARG", "weights must be positive")
        if w > capacity:
            raise BalanceError("SEQ_TOO_LONG", "an item is heavier than the capacity")


def _order(weights):
    """Indices by weight, heaviest first, equal weights in input order."""
    return sorted(range(len(weights)), key=lambda i: (-weights[i], i))


def _ffd_once(weights, capacity, min_groups):
    loads, members = [], []
    for i in _order(weights):
        w = weights[i]
        if len(loads) < min_groups:
            loads.append(w)
            members.append([i])
            continue
        best = -1
        for g in range(len(loads)):  # lightest fitting group, earliest on ties
            if loads[g] + w <= capacity and (best < 0 or loads[g] < loads[best]):
                best = g
        if best < 0:
            loads.append(w)
            members.append([i])
        else:
            loads[best] += w
            members[best].append(i)
    return members


def ffd_allocate(weights, capacity, min_groups=1, divisor=1):
    """Groups (lists of item indices, in creation order) by FFD."""
    weights = [int(w) for w in weights]
    _check(weights, capacity, min_groups, divisor)
    need = min_groups
    while True:
        if need > len(weights):
            raise BalanceError("INVALID_ARG", "more groups required than items")
        groups = _ffd_once(weights, capacity, need)
        g = len(groups)
        if g >= min_groups and g % divisor == 0:
            return groups
        need = -(-max(need, g) // divisor) * divisor  # next multiple of the divisor


def _kk_groups(weights, k):
    """The k-way largest differencing partition (lists of item indices)."""
    # a state: (sets, sums, creation id); sets kept in their current order
    states = []
    for i, w in enumerate(weights):
        sets = [[i]] + [[] for _ in range(k - 1)]
        sums = [w] + [0] * (k - 1)
        states.append((sets, sums, i))
    next_id = len(weights)

    def spread(st):
        return max(st[1]) - min(st[1])

    while len(states) > 1:
        # pop the two states of largest spread (ties: created first)
        states.sort(key=lambda st: (-spread(st), st[2]))
        a, b = states[0], states[1]
        states = states[2:]
        a_desc = sorted(range(k), key=lambda j: (-a[1][j], j))
        b_asc = sorted(range(k), key=lambda j: (b[1][j], j))
        sets = [a[0][a_desc[j]] + b[0][b_asc[j]] for j in range(k)]
        sums = [a[1][a_desc[j]] + b[1][b_asc[j]] for j in range(k)]
        states.append((sets, sums, next_id))
        next_id += 1
    sets, sums, _ = states[0]
    order = sorted(range(k), key=lambda j: (-sums[j], j))
    return [sorted(sets[j]) for j in order]


def kk_allocate(weights, capacity, min_groups=1, divisor=1):
    """(groups, algorithm used): KK, or FFD when a KK group exceeds the capacity."""
    weights = [int(w) for w in weights]
    _check(weights, capacity, min_groups, divisor)
    total = sum(weights)
    k = max(min_groups, -(-total // capacity))
    k = -(-k // divisor) * divisor
    if k > len(weights):
        raise BalanceError("INVALID_ARG", "more groups required than items")
    groups = _kk_groups(weights, k)
    if max(sum(weights[i] for i in g) for g in groups) > capacity:
        return ffd_allocate(weights, capacity, min_groups, divisor), "ffd"
    return groups, "kk"


def group_of(groups, n):
    out = [-1] * n
    for g, members in enumerate(groups):
        for i in members:
            out[i] = g
    return out


@dataclass
class PackingMetrics:
    n_groups: int
    total: int
    max_load: int
    min_load: int
    spread: int
    mean: float
    std_dev: float
    cv: float
    imbalance_ratio: float
    utilization: float
    wasted: int


def packing_metrics(weights, groups, capacity):
    loads = [sum(int(weights[i]) for i in g) for g in groups]
    n = len(loads)
    total = sum(loads)
    mean = total / n
    std = math.sqrt(sum((x - mean) ** 2 for x in loads) / n)
    return PackingMetrics(n_groups=n, total=total, max_load=max(loads), min_load=min(loads),
                          spread=max(loads) - min(loads), mean=mean, std_dev=std,
                          cv=std / mean if mean > 0 else 0.0,
                          imbalance_ratio=max(loads) / mean if mean > 0 else 0.0,
                          utilization=total / (n * capacity), wasted=n * capacity - total)
