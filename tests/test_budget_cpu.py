"""The library's per-layer budget functions (host code in libspin.so, called through the C
ABI with no GPU) against the CPU oracle: bit-exact grid points, and miss curves equal to the
oracle's double-precision values rounded to fp32."""
import random

import numpy as np
import pytest

from oracle import budgets as ob
from sparse_attention_indexer_spin_gb300 import spin


def _batch(rng, n_req, stride, K, ties):
    nbs = [rng.randint(1, stride) for _ in range(n_req)]
    S = np.zeros((n_req, stride), np.float32)
    topk = np.full((n_req, K), -1, np.int32)
    for r, nb in enumerate(nbs):
        S[r, :nb] = [rng.randint(0, 5) if ties else rng.gauss(0, 1) for _ in range(nb)]
        n_valid = rng.randint(0, min(K, nb * 64))
        ids = sorted(rng.sample(range(nb * 64), n_valid))
        topk[r, :n_valid] = ids
    return S, nbs, topk


@pytest.mark.parametrize("seed", range(30))
def test_miss_curve_matches_oracle(seed):
    rng = random.Random(seed)
    n_req, stride, K = rng.randint(1, 5), rng.randint(1, 90), rng.choice([1, 16, 64, 200])
    n_points = rng.choice([2, 3, 11, 21, 101])
    S, nbs, topk = _batch(rng, n_req, stride, K, ties=seed % 2 == 0)
    got = spin.miss_curve(S, nbs, topk, n_points)
    want = ob.mean_miss_curve([S[r].tolist() for r in range(n_req)], nbs,
                              [topk[r].tolist() for r in range(n_req)], K, n_points)
    np.testing.assert_array_equal(got, np.array(want, np.float32))
    assert all(a >= b for a, b in zip(got, got[1:]))  # more budget never misses more


@pytest.mark.parametrize("seed", range(30))
def test_allocation_matches_oracle(seed):
    rng = random.Random(100 + seed)
    L = rng.randint(1, 64)
    n_points = rng.choice([2, 3, 11, 101])
    G = n_points - 1
    miss = np.zeros((L, n_points), np.float32)
    for l in range(L):
        if seed % 3 == 0:   # non-monotone curves are allowed too
            miss[l] = [rng.random() for _ in range(n_points)]
        else:
            vals = sorted((rng.choice([0.0, 0.125, 0.25, 0.5]) if seed % 3 == 1 else rng.random()
                           for _ in range(n_points)), reverse=True)
            miss[l] = vals
    g_min = rng.randint(0, G)
    target = rng.randint(g_min, G)
    g, rho = spin.allocate_budgets(miss, target, g_min)
    want = ob.allocate([[float(v) for v in row] for row in miss], target, g_min)
    assert g.tolist() == want
    assert rho.tolist() == [ob.rho_of(x, n_points) for x in want]
    assert int(g.sum()) == L * target


def test_budget_functions_reject_bad_input():
    S = np.zeros((1, 4), np.float32)
    with pytest.raises(spin.SpinError):
        spin.miss_curve(S, [4], [[0, 1]], 7)           # 6 does not divide 10000
    with pytest.raises(spin.SpinError):
        spin.miss_curve(S, [4], [[0, 4 * 64]], 11)     # id past the context
    with pytest.raises(spin.SpinError):
        spin.miss_curve(S, [5], [[0]], 11)             # nb above the row stride
    S[0, 1] = np.nan
    with pytest.raises(spin.SpinError):
        spin.miss_curve(S, [4], [[0]], 11)
    m = np.zeros((2, 11), np.float32)
    with pytest.raises(spin.SpinError):
        spin.allocate_budgets(m, 3, 4)                 # g_min above the target
    with pytest.raises(spin.SpinError):
        spin.allocate_budgets(m, 11, 0)                # target past the grid
    m[1, 3] = np.nan
    with pytest.raises(spin.SpinError):
        spin.allocate_budgets(m, 5, 0)


def test_uniform_layers_get_the_target():
    curve = np.linspace(1, 0, 101, dtype=np.float32)
    g, rho = spin.allocate_budgets(np.stack([curve] * 21), 60)
    assert g.tolist() == [60] * 21 and rho.tolist() == [4000] * 21


def test_layer_at_the_grid_top_takes_no_spare_point():
    # the worst miss 0.9 needs all 4 points of the first layer and none of the second; both
    # spare points of the total 6 go to the second layer, although the first misses more
    miss = np.array([[1.0, 0.97, 0.95, 0.92, 0.9], [0.5, 0.1, 0.0, 0.0, 0.0]], np.float32)
    g, rho = spin.allocate_budgets(miss, 3)
    assert g.tolist() == [4, 2] and rho.tolist() == [0, 5000]
    assert ob.allocate(miss.astype(np.float64).tolist(), 3, 0) == [4, 2]
