"""CPU oracle of SPIN's per-layer block budgets (plain Python, no numpy tricks).

TEST INFRASTRUCTURE ONLY: imported by tests/, never by the library.

Follows "Sparse Attention Still Has a Dense Problem" (the SPIN project page), section
"Per-layer block budgets" and Figures 5-6: the miss rate of a layer is the fraction of the
dense indexer's top-K slots that fall into skipped blocks; every P steps a dense probe step
measures each layer's miss curve (its miss rate at each budget); the budgets minimise the
worst layer's miss rate while the total budget over all layers stays at the target block
sparsity.  Where the page leaves a step open, these readings are taken:

  - Budgets are kept fractions on a grid of G + 1 points, p_g = g * 10000 / G basis points
    (G divides 10000); layer l keeps p_{g_l}, and sum_l g_l = L * g_target (every layer of
    a request has the same context, so equal weights keep the total kept-block count).
  - The miss curve at kept fraction p is measured against the selection the method makes at
    that budget without its random exploration share: the budget m of the selection's own
    budget rule (10000 - p basis points of sparsity), the forced first and last blocks, then
    the best m - f blocks by predicted block score (equal scores: lower block id).  A larger
    budget selects a superset, so the curve does not increase with p.
  - A layer's curve over a batch is the mean of its requests' curves (each request weighs
    the same); a request with no valid dense top-K slot is left out.
  - The allocation first finds the smallest attainable worst miss tau* and gives each layer
    the fewest grid points reaching miss <= tau*; spare points then go one at a time to the
    layer with the largest miss at its current point (equal misses: the layer with fewer
    points, then the lower index, so flat curves keep the uniform budget; a layer at the top
    of the grid takes none).
"""
from __future__ import annotations

from . import oracle as _o


def miss_curve(S, nb, topk, top_k, n_points):
    """One request's miss curve for one layer.  S: predicted block scores [nb]; topk: the
    dense step's top-K slot ids (-1 = none).  Returns n_points floats."""
    G = n_points - 1
    valid = [int(i) for i in topk if int(i) >= 0]
    f = 2 if nb > 1 else 1
    forced = {0, nb - 1}
    free = sorted((j for j in range(nb) if j not in forced), key=lambda j: (-float(S[j]), j))
    out = []
    for g in range(n_points):
        keep_bp = g * 10000 // G
        m = _o.budget(nb, top_k, 10000 - keep_bp)
        chosen = set(forced) | set(free[: max(m - f, 0)])
        missed = sum(1 for i in valid if i // 64 not in chosen)
        out.append(missed / len(valid) if valid else 0.0)
    return out


def mean_miss_curve(S_rows, nbs, topks, top_k, n_points):
    """The batch's curve for one layer: the mean over requests of miss_curve (requests whose
    dense top-K holds no valid slot are left out; none left gives all zeros)."""
    acc, used = [0.0] * n_points, 0
    for S, nb, topk in zip(S_rows, nbs, topks):
        if not any(int(i) >= 0 for i in topk):
            continue
        c = miss_curve(S, int(nb), topk, top_k, n_points)
        acc = [a + b for a, b in zip(acc, c)]
        used += 1
    return [a / used for a in acc] if used else acc


def allocate(miss, target_g, g_min):
    """Per-layer grid points from the layers' miss curves (a list of equal-length lists)."""
    L = len(miss)
    G = len(miss[0]) - 1
    total = L * target_g

    def need(l, tau):
        for g in range(g_min, G + 1):
            if miss[l][g] <= tau:
                return g
        return None

    taus = sorted({v for row in miss for v in row[g_min:]})
    g = None
    for tau in taus:  # the smallest worst miss whose fewest points fit the total
        cand = [need(l, tau) for l in range(L)]
        if all(c is not None for c in cand) and sum(cand) <= total:
            g = cand
            break
    assert g is not None
    for _ in range(total - sum(g)):
        best = None
        for l in range(L):
            if g[l] >= G:
                continue
            if best is None or (miss[l][g[l]], -g[l]) > (miss[best][g[best]], -g[best]):
                best = l
        g[best] += 1
    return g


def rho_of(g, n_points):
    """Sparsity in basis points of grid point g."""
    return 10000 - g * 10000 // (n_points - 1)
