"""Pins of the per-layer budget oracle (oracle/budgets.py) to facts that do not come from it:
brute-force minimax over every allocation, hand-worked examples, closed forms and the
properties the page fixes (the total budget is kept; the worst layer's miss is minimised).
"""
import itertools
import random

import pytest

from oracle import budgets as ob
from oracle import oracle as o


def _monotone_curve(rng, G, levels=None):
    """A random non-increasing curve from 1 down to 0 on G + 1 points."""
    vals = sorted((rng.choice(levels) if levels else rng.random() for _ in range(G - 1)), reverse=True)
    return [1.0] + vals + [0.0]


@pytest.mark.parametrize("seed", range(40))
def test_allocation_is_minimax_by_brute_force(seed):
    rng = random.Random(seed)
    L, G = rng.randint(1, 4), rng.randint(1, 6)
    levels = [0.0, 0.25, 0.5, 0.75] if seed % 2 else None  # many equal values half the time
    miss = [_monotone_curve(rng, G, levels) for _ in range(L)]
    g_min = rng.randint(0, G)
    target = rng.randint(g_min, G)
    g = ob.allocate(miss, target, g_min)
    assert sum(g) == L * target
    assert all(g_min <= x <= G for x in g)
    best = min(max(miss[l][a[l]] for l in range(L))
               for a in itertools.product(range(g_min, G + 1), repeat=L) if sum(a) == L * target)
    assert max(miss[l][g[l]] for l in range(L)) == best


def test_allocation_hand_example():
    # tau = 0.3 is the smallest worst miss within 4 points (A at 2, B at 1); the spare point
    # goes to B, whose miss 0.3 is the larger one.
    A = [1.0, 0.5, 0.2, 0.1, 0.0]
    B = [1.0, 0.3, 0.3, 0.3, 0.0]
    assert ob.allocate([A, B], 2, 0) == [2, 2]
    # equal curves share the budget equally
    assert ob.allocate([A, A, A], 3, 0) == [3, 3, 3]
    # a layer that never misses takes the floor; the others take the rest
    Z = [0.0] * 5
    assert ob.allocate([Z, A], 2, 1) == [1, 3]
    # flat curves (no miss anywhere) keep the uniform budget: spare points go round the
    # layers with the fewest points
    assert ob.allocate([Z, Z, Z], 2, 0) == [2, 2, 2]
    assert ob.allocate([Z, Z, Z, Z], 3, 1) == [3, 3, 3, 3]
    # equal misses at different points: the layer with fewer points first
    C = [1.0, 0.5, 0.5, 0.5, 0.0]
    assert ob.allocate([C, C], 1, 0) == [1, 1]
    # a layer at the top of the grid takes no spare point, even with the largest miss: the
    # worst miss 0.9 needs all 3 points of the first layer and none of the second; the one
    # spare point of the total 4 goes to the second layer
    assert ob.allocate([[1.0, 0.95, 0.92, 0.9], [0.5, 0.1, 0.0, 0.0]], 2, 0) == [3, 1]


def test_rho_of_grid():
    assert ob.rho_of(0, 101) == 10000 and ob.rho_of(100, 101) == 0 and ob.rho_of(60, 101) == 4000


def test_miss_curve_hand_example():
    # 6 blocks, K = 4 dense top-K slots in blocks 0 (forced), 2 and 3 (two slots).  Ranking by
    # S: 3, 1, 2, 4.  Budget rule with K = 4: at least one block; keep 50 % of 6 -> 3 blocks.
    S = [9.0, 5.0, 1.0, 8.0, 0.5, 9.0]
    topk = [10, 130, 200, 201]
    G = 2  # kept fractions 0, 50 %, 100 %
    curve = ob.miss_curve(S, 6, topk, 4, G + 1)
    # 0 %: budget 1 -> only the forced blocks {0, 5}: slots in 2 and 3 missed (3 of 4)
    # 50 %: budget 3 -> forced + best 1 = block 3: block 2 missed (1 of 4)
    # 100 %: every block
    assert curve == [0.75, 0.25, 0.0]


def test_miss_curve_ties_go_to_the_lower_block():
    # Blocks 1 and 2 tie at the best predicted score; the dense top-K lies in block 2 only.
    # At 50 % (budget 3: the forced blocks 0 and 5 plus one) the method's ranking takes the
    # lower block of a tie, block 1, so every top-K slot is missed; at 100 % none is.
    S = [0.0, 7.0, 7.0, 1.0, 0.5, 0.0]
    topk = [130, 131, 140, 150]
    assert ob.miss_curve(S, 6, topk, 4, 3) == [1.0, 1.0, 0.0]
    # the same context with the top-K in block 1 is fully covered from 50 % on
    assert ob.miss_curve(S, 6, [70, 71, 80, 90], 4, 3) == [1.0, 0.0, 0.0]


def test_miss_curve_closed_form_when_ranking_follows_counts():
    rng = random.Random(3)
    nb, K = 40, 64
    counts = [0] * nb
    slots = []
    while len(slots) < K:
        j = rng.randrange(1, nb - 1)
        s = j * 64 + rng.randrange(64)
        if s not in slots:
            slots.append(s)
            counts[j] += 1
    S = [counts[j] + j * 1e-3 for j in range(nb)]  # distinct, ordered by count
    G = 20
    curve = ob.miss_curve(S, nb, sorted(slots), K, G + 1)
    order = sorted(range(1, nb - 1), key=lambda j: -S[j])
    for g in range(G + 1):
        m = o.budget(nb, K, 10000 - g * 10000 // G)
        kept = sum(counts[j] for j in order[: max(m - 2, 0)])
        assert curve[g] == pytest.approx(1.0 - kept / K, abs=0)
    assert all(a >= b for a, b in zip(curve, curve[1:]))
    assert curve[-1] == 0.0


def test_miss_curve_forced_only_and_empty():
    # every dense top-K slot in the forced blocks: nothing is ever missed
    assert ob.miss_curve([1.0] * 10, 10, [0, 1, 9 * 64 + 3], 3, 11) == [0.0] * 11
    # no valid top-K slot: defined as no miss
    assert ob.miss_curve([1.0] * 10, 10, [-1, -1], 2, 3) == [0.0] * 3


def test_mean_curve_of_identical_requests_and_skips_empty():
    S = [9.0, 5.0, 1.0, 8.0, 0.5, 9.0]
    topk = [10, 130, 200, 201]
    one = ob.miss_curve(S, 6, topk, 4, 3)
    assert ob.mean_miss_curve([S, S, S], [6, 6, 6], [topk, topk, topk], 4, 3) == one
    # a request with no valid slot does not count; two different requests average
    other = ob.miss_curve(S, 6, [10, 11, 12, 13], 4, 3)  # all in forced block 0: no miss
    assert other == [0.0, 0.0, 0.0]
    got = ob.mean_miss_curve([S, S, S], [6, 6, 6], [topk, [-1] * 4, [10, 11, 12, 13]], 4, 3)
    assert got == [(a + b) / 2 for a, b in zip(one, other)]
    assert ob.mean_miss_curve([S], [6], [[-1] * 4], 4, 3) == [0.0, 0.0, 0.0]
