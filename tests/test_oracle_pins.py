"""Pins of the CPU oracle against what the paper and the mathematics fix.

Each test checks an oracle function against something other than the oracle itself:
a library routine (numpy's Philox, torch's number-format conversions, numpy
reductions, sorts and einsum), a closed form, an invariant stated by the paper, a
hand-derived table (tests/golden/), or brute force on tiny inputs.

Paper: "SPIN: Shadow Predictive Indexer for Sparse Attention" (arXiv 2610.09025).
"""
import math
import os

import numpy as np
import pytest
import torch

from sparse_attention_indexer_spin_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append([int(x) for x in line.split()])
    return rows


def tiny_cfg(o, **kw):
    base = dict(n_req=2, max_slots=300, max_rows=4, n_heads=2, head_dim=4, kv_heads=2,
                q_dtype="f32", k_dtype="f32", top_k=16, rho_bp=4000, gamma_bp=500,
                alpha=0.9, combine="max", seed=7)
    base.update(kw)
    return o.make_cfg(**base)


# --------------------------------------------------------------------------- Philox

def _numpy_philox(ctr, key):
    """numpy's Philox4x64-10 advances its 256-bit counter before each block; start one
    below the wanted counter."""
    c = list(ctr)
    for i in range(4):  # 256-bit decrement (the all-zero counter wraps to all ones)
        if c[i] != 0:
            c[i] -= 1
            break
        c[i] = (1 << 64) - 1
    bg = np.random.Philox(key=np.array(key, dtype=np.uint64))
    st = bg.state
    st["state"]["counter"] = np.array(c, dtype=np.uint64)
    st["buffer_pos"] = 4
    bg.state = st
    return [int(x) for x in bg.random_raw(4)]


@pytest.mark.parametrize("ctr,key", [
    ([1, 0, 0, 0], [0, 0]),
    ([5, 0, 3, 17], [0x0123456789ABCDEF, 42]),
    ([0, 1, 0, 0], [7, 0]),                      # exercises the counter carry in numpy
    ([2**64 - 1, 2**63, 99, 2**40], [2**64 - 1, 2**64 - 1]),
    ([123456, 3, 95, 2047], [2026, 1]),
])
def test_philox_matches_numpy(oracle_mod, ctr, key):
    assert oracle_mod.philox4x64_10(ctr, key) == _numpy_philox(ctr, key)


def test_explore_keys_are_the_halves_of_one_philox_output(oracle_mod):
    """Blocks 8m .. 8m+7 take the eight 32-bit halves of the output for counter m, word by
    word, high half first."""
    m = 37
    out = oracle_mod.philox4x64_10([11, 2, 5, m], [99, 3])
    halves = []
    for w in out:
        halves += [w >> 32, w & 0xFFFFFFFF]
    assert [oracle_mod.explore_key(99, 3, 11, 2, 5, 8 * m + h) for h in range(8)] == halves
    # the next counter serves the next eight blocks
    out2 = oracle_mod.philox4x64_10([11, 2, 5, m + 1], [99, 3])
    assert oracle_mod.explore_key(99, 3, 11, 2, 5, 8 * m + 8) == out2[0] >> 32


# --------------------------------------------------------------------- number formats

def test_e4m3_decode_all_codes(oracle_mod):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    for code in range(256):
        got = oracle_mod.decode_e4m3(code)
        want = float(ref[code])
        if math.isnan(want):
            assert math.isnan(got)
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), code


def test_bf16_decode(oracle_mod):
    rng = np.random.default_rng(0)
    bits = np.concatenate([np.arange(0, 65536, 97), rng.integers(0, 65536, 4000)]).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64)
    for b, r in zip(bits.tolist(), ref.tolist()):
        got = oracle_mod.decode_bf16(b)
        if math.isnan(r):
            assert math.isnan(got)
        else:
            assert got == r


# ---------------------------------------------------------------- budget, exploration

@pytest.mark.parametrize("row", _table("budget_table.txt"))
def test_budget_table(oracle_mod, row):
    B, K, rho, m = row
    assert oracle_mod.budget(B, K, rho) == m


@pytest.mark.parametrize("row", _table("explore_count_table.txt"))
def test_explore_count_table(oracle_mod, row):
    m, f, g, e = row
    assert oracle_mod.explore_count(m, f, g) == e


def test_budget_properties(oracle_mod):
    # capped by B, at least min(B, ceil(K/b)), monotone non-increasing in rho
    for B in (1, 2, 7, 64, 65, 1000, 2048):
        for K in (1, 64, 256, 2048):
            prev = None
            for rho in range(0, 10001, 250):
                m = oracle_mod.budget(B, K, rho)
                assert 1 <= m <= B
                assert m >= min(B, -(-K // 64))
                assert m >= min(B, -(-(10000 - rho) * B // 10000))
                if prev is not None:
                    assert m <= prev
                prev = m
            assert oracle_mod.budget(B, K, 0) == B


# ------------------------------------------------------------------- block scores

def _blockwise_max(x, n):
    starts = np.arange(0, n, 64)
    return np.maximum.reduceat(x[:n], starts)


@pytest.mark.parametrize("n", [1, 63, 64, 65, 130, 257])
def test_block_scores_reduce_to_vertical_max(oracle_mod, n):
    """D = -inf everywhere: Eq. 1 gives V[i], Eq. 2 the blockwise max of V."""
    cfg = tiny_cfg(oracle_mod)
    rng = np.random.default_rng(n)
    V = rng.standard_normal(cfg.max_slots).astype(np.float32)
    D = np.full(oracle_mod.d_len(cfg), -np.inf, dtype=np.float32)
    q = n - 1 + 2
    S = oracle_mod.block_scores(cfg, V, D, n, q)
    np.testing.assert_array_equal(S, _blockwise_max(V, n))


@pytest.mark.parametrize("n", [1, 64, 100, 257])
def test_block_scores_reduce_to_diagonal_max(oracle_mod, n):
    """V = -inf: S[j] is the max of D over the offsets q - i of block j's slots."""
    cfg = tiny_cfg(oracle_mod)
    rng = np.random.default_rng(100 + n)
    V = np.full(cfg.max_slots, -np.inf, dtype=np.float32)
    D = rng.standard_normal(oracle_mod.d_len(cfg)).astype(np.float32)
    q = n + 1
    S = oracle_mod.block_scores(cfg, V, D, n, q)
    diag = D[q - np.arange(n)]              # value seen by slot i
    np.testing.assert_array_equal(S, _blockwise_max(diag, n))


def test_block_scores_sum_mode_with_zero_diagonal(oracle_mod):
    cfg = tiny_cfg(oracle_mod, combine="sum")
    rng = np.random.default_rng(3)
    V = rng.standard_normal(cfg.max_slots).astype(np.float32)
    D = np.zeros(oracle_mod.d_len(cfg), dtype=np.float32)
    S = oracle_mod.block_scores(cfg, V, D, 200, 205)
    np.testing.assert_array_equal(S, _blockwise_max(V, 200))


def test_block_scores_brute_force_tiny(oracle_mod):
    """Brute force over a 3-block context (one block partial), both combiners."""
    for combine in ("max", "sum"):
        cfg = tiny_cfg(oracle_mod, combine=combine)
        rng = np.random.default_rng(9)
        n, q = 150, 152
        V = rng.standard_normal(cfg.max_slots).astype(np.float32)
        D = rng.standard_normal(oracle_mod.d_len(cfg)).astype(np.float32)
        S = oracle_mod.block_scores(cfg, V, D, n, q)
        assert len(S) == 3
        for j in range(3):
            vals = []
            for i in range(64 * j, min(64 * (j + 1), n)):
                a, b = float(V[i]), float(D[q - i])
                vals.append(max(a, b) if combine == "max" else float(np.float32(a) + np.float32(b)))
            assert S[j] == max(vals)


# ------------------------------------------------------------------- selection

def _random_state(o, cfg, rng, warm=1):
    V = rng.standard_normal((cfg.n_req, cfg.max_slots)).astype(np.float32)
    D = rng.standard_normal((cfg.n_req, o.d_len(cfg))).astype(np.float32)
    return V, D, np.full(cfg.n_req, warm, dtype=np.int32)


def _numpy_explore_keys(seed, layer, step, row, req, js):
    """Exploration draws from numpy's own Philox4x64-10: block j takes 32-bit half j % 8
    (word by word, high half first) of the output for counter (step, row, req, j // 8)
    under key (seed, layer)."""
    cache, out = {}, []
    for j in js:
        m = int(j) // 8
        if m not in cache:
            cache[m] = _numpy_philox([step, row, req, m], [seed, layer])
        w = cache[m][(int(j) % 8) // 2]
        out.append((w >> 32) if j % 2 == 0 else (w & 0xFFFFFFFF))
    return out


def _check_selection(o, cfg, V, D, n, q, sel, rho_bp, row=0, explore=None):
    """Invariants of §3.2 / §3.2.1 against an independent numpy ranking.  With
    explore = (seed, layer, step, req) the explored blocks must also be the e blocks left
    outside the forced and top blocks with the smallest draws (lower j on equal draws)."""
    B = -(-n // 64)
    m = o.budget(B, cfg.top_k, rho_bp)
    f = 2 if B > 1 else 1
    e = o.explore_count(m, f, cfg.gamma_bp)
    t = max(m - f - e, 0) if m > f else 0
    assert len(sel) == max(m, f)
    assert list(sel) == sorted(set(sel))
    assert 0 in sel and (B - 1) in sel
    S = o.block_scores(cfg, V, D, n, q + row)
    free = np.array([j for j in range(B) if j not in (0, B - 1)], dtype=np.int64)
    order = free[np.lexsort((free, -S[free].astype(np.float64)))]
    top = set(order[:t].tolist())
    assert top <= set(sel)
    explored = set(sel) - top - {0, B - 1}
    assert len(explored) == (e if m > f else 0)
    assert not (explored & top)
    if explore is not None and m > f:
        seed, layer, step, req = explore
        rest = [j for j in free.tolist() if j not in top]
        keys = _numpy_explore_keys(seed, layer, step, row, req, rest)
        want = sorted(zip(keys, rest))[:e]
        assert explored == {j for _, j in want}
    return top, explored


@pytest.mark.parametrize("n,rho", [(4096, 4000), (4100, 4000), (130, 4000), (2000, 2000),
                                   (640, 9000), (64, 4000), (65, 5000)])
def test_selection_invariants(oracle_mod, n, rho):
    o = oracle_mod
    cfg = tiny_cfg(o, n_req=3, max_slots=4200, top_k=256 if n > 1000 else 64, gamma_bp=1000)
    rng = np.random.default_rng(n + rho)
    V, D, warm = _random_state(o, cfg, rng)
    n_slots = np.array([n, max(1, n - 37), n], dtype=np.int32)
    q_pos = n_slots - 1
    q_pos[2] += 3
    blocks, nb, _, _, ok = o.select_blocks(cfg, V, D, warm, n_slots, q_pos, 1, rho, 5, 2)
    assert ok
    for r in range(cfg.n_req):
        sel = blocks[r, 0, : nb[r, 0]]
        _check_selection(o, cfg, V[r], D[r], int(n_slots[r]), int(q_pos[r]), sel, rho,
                         explore=(7, 2, 5, r))


def test_reset_of_one_request_leaves_the_others(oracle_mod):
    """A reset (§3.2: a request starts cold, and its first step is dense) clears that request's
    V, D and warm flag only; req = -1 clears every request."""
    o = oracle_mod
    cfg = o.make_cfg(n_req=3, max_slots=256, max_rows=2, n_heads=2, head_dim=4, kv_heads=2,
                     q_dtype="f32", k_dtype="f32", top_k=16, rho_bp=4000, gamma_bp=500, alpha=0.5)
    rng = np.random.default_rng(5)
    V, D, warm = o.new_state(cfg)
    V[:] = rng.random(V.shape) + 1
    D[:] = rng.random(D.shape) + 1
    warm[:] = 1
    V0, D0 = V.copy(), D.copy()
    o.init_state(cfg, V, D, warm, 1)
    assert np.all(V[1] == 0) and np.all(D[1] == 0) and warm[1] == 0
    for r in (0, 2):
        assert np.array_equal(V[r], V0[r]) and np.array_equal(D[r], D0[r]) and warm[r] == 1
    o.init_state(cfg, V, D, warm)
    assert not V.any() and not D.any() and not warm.any()


def test_rho_zero_and_cold_are_dense(oracle_mod):
    o = oracle_mod
    cfg = tiny_cfg(o, n_req=2, max_slots=2000, top_k=64)
    rng = np.random.default_rng(1)
    V, D, warm = _random_state(o, cfg, rng)
    n_slots = np.array([1999, 777], dtype=np.int32)
    blocks, nb, _, _, ok = o.select_blocks(cfg, V, D, warm, n_slots, n_slots - 1, 1, 0)
    assert ok
    for r in range(2):
        B = -(-int(n_slots[r]) // 64)
        assert list(blocks[r, 0, : nb[r, 0]]) == list(range(B))
    warm[:] = 0
    blocks, nb, _, _, ok = o.select_blocks(cfg, V, D, warm, n_slots, n_slots - 1, 1, 6000)
    for r in range(2):
        B = -(-int(n_slots[r]) // 64)
        assert list(blocks[r, 0, : nb[r, 0]]) == list(range(B))


def test_exploration_uniform_chi_square(oracle_mod):
    """Random exploration picks e distinct blocks uniformly among the non-selected ones:
    frequencies over many steps against e / (#candidates), chi-square at p = 1e-4."""
    o = oracle_mod
    n = 64 * 60
    cfg = tiny_cfg(o, n_req=1, max_slots=n + 8, top_k=64, gamma_bp=2000)
    V = np.linspace(0, 1, cfg.max_slots, dtype=np.float32)[None, :].copy()  # fixed ranking
    D = np.full((1, o.d_len(cfg)), -1e30, dtype=np.float32)
    warm = np.ones(1, dtype=np.int32)
    ns = np.array([n], dtype=np.int32)
    counts = np.zeros(60)
    steps = 3000
    top = None
    for s in range(steps):
        blocks, nb, _, _, ok = o.select_blocks(cfg, V, D, warm, ns, ns - 1, 1, 5000, s, 0)
        t, ex = _check_selection(o, cfg, V[0], D[0], n, n - 1, blocks[0, 0, : nb[0, 0]], 5000,
                                 explore=(7, 0, s, 0) if s < 50 else None)
        top = t if top is None else top
        assert t == top
        for j in ex:
            counts[j] += 1
    cand = [j for j in range(1, 59) if j not in top]
    e = o.explore_count(o.budget(60, 64, 5000), 2, 2000)
    expected = steps * e / len(cand)
    chi2 = float(((counts[cand] - expected) ** 2 / expected).sum())
    from scipy.stats import chi2 as chi2_dist
    assert chi2 < chi2_dist.ppf(1 - 1e-4, len(cand) - 1), chi2
    assert counts[list(top)].sum() == 0


def test_union_is_or_of_rows(oracle_mod):
    o = oracle_mod
    cfg = tiny_cfg(o, n_req=2, max_slots=3000, top_k=128, max_rows=4)
    rng = np.random.default_rng(5)
    V, D, warm = _random_state(o, cfg, rng)
    ns = np.array([2900, 1500], dtype=np.int32)
    blocks, nb, union, nu, ok = o.select_blocks(cfg, V, D, warm, ns, ns - 1, 4, 4000, 3, 1)
    assert ok
    for r in range(2):
        rows = [set(blocks[r, k, : nb[r, k]].tolist()) for k in range(4)]
        for k in range(4):
            _check_selection(o, cfg, V[r], D[r], int(ns[r]), int(ns[r] - 1),
                             blocks[r, k, : nb[r, k]], 4000, row=k, explore=(7, 1, 3, r))
        assert list(union[r, : nu[r]]) == sorted(set().union(*rows))
        assert nu[r] >= nb[r, 0]


def test_invalid_request_is_skipped(oracle_mod):
    o = oracle_mod
    cfg = tiny_cfg(o, n_req=2, max_slots=500)
    V, D, warm = o.new_state(cfg)
    ns = np.array([400, 400], dtype=np.int32)
    qp = np.array([399, 10], dtype=np.int32)       # request 1: q < N - 1
    blocks, nb, _, _, ok = o.select_blocks(cfg, V, D, warm, ns, qp, 1)
    assert not ok and nb[1, 0] == 0 and nb[0, 0] == 7


# ------------------------------------------------------------------------- scores

def _decode_torch(raw, dtype):
    if dtype == "f32":
        return raw.astype(np.float64)
    if dtype == "bf16":
        return torch.from_numpy(raw.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    return torch.from_numpy(raw.copy()).view(torch.float8_e4m3fn).double().numpy()


def _brute_scores(cfg_kw, q, w, pool, scale, bt, blist, nlist, ns, rows):
    """Dense numpy einsum in float64 over torch-decoded inputs."""
    H, d, kvh = cfg_kw["n_heads"], cfg_kw["head_dim"], cfg_kw["kv_heads"]
    qd = _decode_torch(q, cfg_kw["q_dtype"]).reshape(q.shape[0], rows, H, d)
    kd = _decode_torch(pool, cfg_kw["k_dtype"]).reshape(pool.shape[0], 64, kvh, d)
    R, MB = bt.shape[0], blist.shape[1]
    out = np.zeros((R, rows, MB * 64))
    for r in range(R):
        for k in range(nlist[r]):
            blk = blist[r, k]
            page = bt[r, blk]
            keys = kd[page]                                   # [64][kvh][d]
            if kvh == 1:
                keys = np.broadcast_to(keys, (64, H, d))
            dots = np.einsum("shc,xhc->xsh", keys, qd[r])      # [rows][64][H]
            if scale is not None:
                dots = dots * scale[page][None, :, None].astype(np.float64)
            z = (np.maximum(dots, 0) * w[r][:, None, :].astype(np.float64)).sum(-1)
            valid = (blk * 64 + np.arange(64)) < ns[r]
            out[r, :, k * 64:(k + 1) * 64] = np.where(valid[None, :], z, 0.0)
    return out


@pytest.mark.parametrize("qd,kd,kvh,rows", [("f32", "f32", 2, 1), ("bf16", "bf16", 2, 3),
                                             ("bf16", "e4m3", 1, 1), ("f32", "bf16", 1, 4),
                                             ("bf16", "e4m3", 2, 2)])
def test_scores_brute_force_tiny(oracle_mod, qd, kd, kvh, rows):
    o = oracle_mod
    kw = dict(n_req=2, max_slots=200, max_rows=4, n_heads=2, head_dim=4, kv_heads=kvh,
              q_dtype=qd, k_dtype=kd, top_k=16, rho_bp=0, gamma_bp=0, alpha=0.5)
    cfg = o.make_cfg(**kw)
    wl = syn.Workload("tiny", n_req=2, n_layers=1, n0=130, n_heads=2, head_dim=4,
                      kv_heads=kvh, q_dtype=qd, k_dtype=kd, top_k=16, rho_bp=0, gamma_bp=0,
                      alpha=0.5, steps=4, rows=rows, heavy=3, rope_dims=2, shuffle=True,
                      mean_accept=2.0 if rows > 1 else 0.0)
    inp = syn.SyntheticInputs(wl, "cpu")
    cfg = o.make_cfg(**{**kw, "max_slots": wl.max_slots})
    q, w, qp = inp.step_inputs()
    qn, wn = syn.raw_numpy(q), w.numpy()
    pool = syn.raw_numpy(inp.k_pool[0])
    scale = None if inp.k_scale[0] is None else inp.k_scale[0].numpy()
    bt = inp.block_table.numpy()
    MB = o.max_blocks(cfg)
    ns = np.array([130, 67], dtype=np.int32)
    blist = np.full((2, MB), -1, dtype=np.int32)
    blist[0, :3] = [0, 1, 2]
    blist[1, :2] = [0, 1]
    nlist = np.array([3, 2], dtype=np.int32)
    sc, mags, ok = o.indexer_score(cfg, qn, wn, pool, scale, bt, blist, nlist, ns, rows,
                                   want_mags=True)
    assert ok
    ref = _brute_scores(kw, qn, wn, pool, scale, bt, blist, nlist, ns, rows)
    np.testing.assert_allclose(sc.astype(np.float64), ref, rtol=0, atol=1e-6 * (1 + mags.max()))
    assert np.all(mags * (1 + 2.0 ** -23) >= np.abs(sc))   # |z| <= magnitude, up to float rounding


def test_scores_integer_inputs_exact(oracle_mod):
    """Integer-valued q, k, w: every sum is exact, so the float result equals numpy's."""
    o = oracle_mod
    kw = dict(n_req=1, max_slots=192, max_rows=2, n_heads=3, head_dim=8, kv_heads=3,
              q_dtype="f32", k_dtype="f32", top_k=8, rho_bp=0, gamma_bp=0, alpha=0.5)
    cfg = o.make_cfg(**kw)
    rng = np.random.default_rng(4)
    q = rng.integers(-4, 5, (1, 2, 3, 8)).astype(np.float32)
    w = rng.integers(-2, 4, (1, 2, 3)).astype(np.float32)
    pool = rng.integers(-5, 6, (3, 64, 3, 8)).astype(np.float32)
    bt = np.array([[2, 0, 1]], dtype=np.int32)
    blist = np.array([[0, 1, 2]], dtype=np.int32)
    ns = np.array([150], dtype=np.int32)
    sc, ok = o.indexer_score(cfg, q, w, pool, None, bt, blist, np.array([3], np.int32), ns, 2)
    ref = _brute_scores(kw, q, w, pool, None, bt, blist, np.array([3]), ns, 2)
    np.testing.assert_array_equal(sc.astype(np.float64), ref)


def test_scores_fp8_scale_sign_and_scaling(oracle_mod):
    """The per-slot FP8 scale multiplies the dot product before the ReLU (§2 with per-slot
    key scales).  Pinned without retyping the score: since ReLU(x) - ReLU(-x) = x, scoring
    with scales s and -s differs by sum_h w_h s (q_h . k), a plain numpy dot product with no
    ReLU; and doubling every scale doubles every score exactly."""
    o = oracle_mod
    kw = dict(n_req=1, max_slots=128, max_rows=1, n_heads=4, head_dim=16, kv_heads=1,
              q_dtype="bf16", k_dtype="e4m3", top_k=8, rho_bp=0, gamma_bp=0, alpha=0.5)
    cfg = o.make_cfg(**kw)
    rng = np.random.default_rng(11)
    q = rng.integers(0, 65535, (1, 1, 4, 16)).astype(np.uint16) & 0xBFFF   # finite bf16, both signs
    w = rng.random((1, 1, 4)).astype(np.float32)
    pool = rng.integers(0, 255, (2, 64, 1, 16)).astype(np.uint8)
    pool[(pool & 0x7F) == 0x7F] = 0x01                                       # no NaN codes
    scale = (rng.random((2, 64)) * 2 - 1).astype(np.float32)                 # signed scales
    bt = np.array([[1, 0]], dtype=np.int32)
    args = (bt, np.array([[0, 1]], np.int32), np.array([2], np.int32), np.array([128], np.int32), 1)
    zp, mp, ok1 = o.indexer_score(cfg, q, w, pool, scale, *args, want_mags=True)
    zn, _, ok2 = o.indexer_score(cfg, q, w, pool, -scale, *args, want_mags=True)
    z2, ok3 = o.indexer_score(cfg, q, w, pool, 2 * scale, *args)
    assert ok1 and ok2 and ok3
    qd = _decode_torch(q, "bf16").reshape(4, 16)
    kd = _decode_torch(pool, "e4m3").reshape(2, 64, 16)
    lin = np.zeros(128)
    for i in range(128):
        page, s = bt[0, i // 64], i % 64
        lin[i] = float(scale[page, s]) * float(np.dot(w[0, 0].astype(np.float64), qd @ kd[page, s]))
    diff = zp[0, 0].astype(np.float64) - zn[0, 0].astype(np.float64)
    np.testing.assert_allclose(diff, lin, rtol=0, atol=1e-6 * (1 + 2 * mp.max()))
    assert np.any(zp[0, 0] > 0) and np.any(zn[0, 0] > 0) and np.any(lin < 0) and np.any(lin > 0)
    np.testing.assert_array_equal(z2, 2 * zp)


def test_score_slot_matches_block_scores(oracle_mod):
    o = oracle_mod
    kw = dict(n_req=1, max_slots=128, max_rows=1, n_heads=4, head_dim=16, kv_heads=1,
              q_dtype="bf16", k_dtype="e4m3", top_k=8, rho_bp=0, gamma_bp=0, alpha=0.5)
    cfg = o.make_cfg(**kw)
    rng = np.random.default_rng(2)
    q = rng.integers(0, 65535, (1, 1, 4, 16)).astype(np.uint16) & 0xBFFF   # finite bf16
    w = rng.random((1, 1, 4)).astype(np.float32)
    pool = rng.integers(0, 126, (2, 64, 1, 16)).astype(np.uint8)
    scale = rng.random((2, 64)).astype(np.float32)
    bt = np.array([[1, 0]], dtype=np.int32)
    sc, ok = o.indexer_score(cfg, q, w, pool, scale, bt, np.array([[0, 1]], np.int32),
                             np.array([2], np.int32), np.array([128], np.int32), 1)
    for i in (0, 5, 63, 64, 127):
        page, s = bt[0, i // 64], i % 64
        z, _ = o.score_slot(cfg, q[0], w[0], pool[page, s], scale[page, s], 1)
        assert z[0] == sc[0, 0, i]


# -------------------------------------------------------------------------- top-K

def test_topk_brute_force_with_ties(oracle_mod):
    o = oracle_mod
    cfg = tiny_cfg(o, n_req=2, max_slots=700, top_k=50)
    MB = o.max_blocks(cfg)
    rng = np.random.default_rng(8)
    rows = 2
    scores = np.round(rng.standard_normal((2, rows, MB * 64)) * 3).astype(np.float32)
    scores[scores == 0] = -0.0                     # -0 and +0 compare equal
    blist = np.full((2, MB), -1, dtype=np.int32)
    sel0 = np.array([0, 2, 3, 7, 10])
    blist[0, :5] = sel0
    blist[1, :2] = [0, 1]
    nlist = np.array([5, 2], dtype=np.int32)
    ns = np.array([680, 100], dtype=np.int32)
    idx, ok = o.topk(cfg, scores, blist, nlist, ns, rows)
    assert ok
    for r in range(2):
        for row in range(rows):
            ids, vals = [], []
            for k in range(nlist[r]):
                for s in range(64):
                    i = blist[r, k] * 64 + s
                    if i < ns[r]:
                        ids.append(i)
                        vals.append(scores[r, row, k * 64 + s])
            ids, vals = np.array(ids), np.array(vals, dtype=np.float64)
            order = np.lexsort((ids, -vals))[: cfg.top_k]
            want = np.sort(ids[order])
            want = np.concatenate([want, -np.ones(cfg.top_k - len(want), dtype=np.int64)])
            np.testing.assert_array_equal(idx[r, row], want)
    assert (idx[1, 0] >= 0).sum() == 50 and (idx[1, 0, :] < 100).all()


def test_topk_pads_when_few_slots(oracle_mod):
    o = oracle_mod
    cfg = tiny_cfg(o, n_req=1, max_slots=200, top_k=100)
    MB = o.max_blocks(cfg)
    scores = np.arange(MB * 64, dtype=np.float32)[None, None, :]
    blist = np.zeros((1, MB), dtype=np.int32)
    idx, ok = o.topk(cfg, scores, blist, np.array([1], np.int32), np.array([40], np.int32))
    np.testing.assert_array_equal(idx[0, 0, :40], np.arange(40))
    assert (idx[0, 0, 40:] == -1).all()


# ---------------------------------------------------------------------------- EMA

def test_ema_closed_form_constant_observation(oracle_mod):
    """n equal observations z from V0: V_n = a^n V0 + (1 - a^n) z (exact in reals)."""
    o = oracle_mod
    for alpha in (0.5, 0.9):
        cfg = tiny_cfg(o, n_req=1, max_slots=128, alpha=alpha)
        MB = o.max_blocks(cfg)
        V, D, warm = o.new_state(cfg)
        rng = np.random.default_rng(1)
        V0 = rng.standard_normal(V.shape).astype(np.float32)
        V[:] = V0
        z = rng.standard_normal(MB * 64).astype(np.float32)
        blist = np.array([[0, 1]], dtype=np.int32)
        ns = np.array([128], np.int32)
        for step in range(1, 41):
            D[:] = 0
            assert o.replay_ema(cfg, V, D, warm, z[None, None, :], blist,
                                np.array([2], np.int32), ns, np.array([127], np.int32))
            a_n = np.float64(alpha) ** step
            want = a_n * V0.astype(np.float64) + (1 - a_n) * z.astype(np.float64)
            err = np.abs(V.astype(np.float64) - want)
            scale = np.abs(V0).astype(np.float64) + np.abs(z).astype(np.float64)
            assert (err <= 4 * step * 2.0 ** -24 * scale + 1e-30).all()
            # D: one observation from 0: (1 - a) z at offset q - i
            dwant = (1 - np.float64(np.float32(alpha))) * z.astype(np.float64)
            np.testing.assert_allclose(D[0, 127 - np.arange(128)], dwant, rtol=2e-7, atol=0)
        assert warm[0] == 1


def test_mtp_replay_closed_form_and_prefix(oracle_mod):
    """Prefix-valid replay (§3.2.2): after rows 0..a,
    V = a^(a+1) V0 + (1-a) sum_r a^(a-r) z_r; rows above a leave no trace."""
    o = oracle_mod
    cfg = tiny_cfg(o, n_req=3, max_slots=256, alpha=0.9, max_rows=4)
    MB = o.max_blocks(cfg)
    rng = np.random.default_rng(12)
    V0 = rng.standard_normal((3, cfg.max_slots)).astype(np.float32)
    D0 = rng.standard_normal((3, o.d_len(cfg))).astype(np.float32)
    scores = rng.standard_normal((3, 4, MB * 64)).astype(np.float32)
    blist = np.full((3, MB), -1, dtype=np.int32)
    blist[:, :2] = [1, 3]
    nlist = np.full(3, 2, dtype=np.int32)
    ns = np.full(3, 250, dtype=np.int32)
    qp = ns - 1
    acc = np.array([0, 2, 3], dtype=np.int32)
    V, D, warm = V0.copy(), D0.copy(), np.zeros(3, np.int32)
    assert o.replay_ema(cfg, V, D, warm, scores, blist, nlist, ns, qp, 4, acc)
    al = np.float64(0.9)
    for r in range(3):
        a = acc[r]
        for k, blk in enumerate(blist[r, :2]):
            for s in range(64):
                i = blk * 64 + s
                if i >= 250:
                    assert V[r, i] == V0[r, i]
                    continue
                zs = [np.float64(scores[r, row, k * 64 + s]) for row in range(a + 1)]
                want = al ** (a + 1) * np.float64(V0[r, i]) + (1 - al) * sum(
                    al ** (a - row) * zs[row] for row in range(a + 1))
                assert abs(V[r, i] - want) <= 1e-6 * (abs(want) + 1)
        untouched = np.ones(cfg.max_slots, bool)
        untouched[64:128] = False
        untouched[192:250] = False
        np.testing.assert_array_equal(V[r, untouched], V0[r, untouched])
        # D closed form: offset o collects rows r' <= a whose slot q + r' - o is scored
        for off in range(0, 260):
            hits = []
            for row in range(a + 1):
                i = qp[r] + row - off
                if 0 <= i < 250 and (i // 64) in (1, 3):
                    k = 0 if i // 64 == 1 else 1
                    hits.append(np.float64(scores[r, row, k * 64 + i % 64]))
            want = np.float64(D0[r, off])
            for h in hits:
                want = al * want + (1 - al) * h
            assert abs(D[r, off] - want) <= 1e-6 * (abs(want) + 1)


def test_replay_a0_equals_single_row(oracle_mod):
    o = oracle_mod
    cfg4 = tiny_cfg(o, n_req=2, max_slots=256, max_rows=4)
    MB = o.max_blocks(cfg4)
    rng = np.random.default_rng(3)
    V0 = rng.standard_normal((2, cfg4.max_slots)).astype(np.float32)
    D0 = rng.standard_normal((2, o.d_len(cfg4))).astype(np.float32)
    scores = rng.standard_normal((2, 4, MB * 64)).astype(np.float32)
    blist = np.tile(np.array([0, 2, 3, 3], np.int32), (2, 1))
    nlist = np.array([3, 2], np.int32)
    ns = np.array([200, 190], np.int32)
    qp = ns - 1
    Va, Da, wa = V0.copy(), D0.copy(), np.zeros(2, np.int32)
    o.replay_ema(cfg4, Va, Da, wa, scores, blist, nlist, ns, qp, 4, np.zeros(2, np.int32))
    Vb, Db, wb = V0.copy(), D0.copy(), np.zeros(2, np.int32)
    o.replay_ema(cfg4, Vb, Db, wb, np.ascontiguousarray(scores[:, :1]), blist, nlist, ns, qp, 1)
    assert Va.tobytes() == Vb.tobytes() and Da.tobytes() == Db.tobytes()


# --------------------------------------------------------------- whole step (rho = 0)

def test_rho_zero_step_equals_dense_topk(oracle_mod):
    """At 0 % target sparsity every block is scored, so SPIN's top-K must equal the dense
    indexer's top-K (integer-valued inputs make both score sets exact)."""
    o = oracle_mod
    rng = np.random.default_rng(21)
    R, H, d, n = 2, 3, 8, 1000
    kw = dict(n_req=R, max_slots=1100, max_rows=1, n_heads=H, head_dim=d, kv_heads=1,
              q_dtype="f32", k_dtype="f32", top_k=100, rho_bp=0, gamma_bp=500, alpha=0.9)
    cfg = o.make_cfg(**kw)
    MB = o.max_blocks(cfg)
    pool = rng.integers(-3, 4, (R * MB, 64, 1, d)).astype(np.float32)
    bt = rng.permutation(R * MB).astype(np.int32).reshape(R, MB)
    V, D, warm = o.new_state(cfg)
    V[:] = rng.standard_normal(V.shape)
    warm[:] = 1
    stepper = o.OracleStep(cfg)
    for step in range(3):
        q = rng.integers(-3, 4, (R, 1, H, d)).astype(np.float32)
        w = rng.integers(0, 3, (R, 1, H)).astype(np.float32)
        ns = np.array([n + step, n - 300 + step], np.int32)
        out = stepper.run(V, D, warm, q, w, pool, None, bt, ns, ns - 1, 1, step)
        assert out["ok"]
        for r in range(R):
            N = int(ns[r])
            keys = pool[bt[r, np.arange(N) // 64], np.arange(N) % 64, 0]      # [N][d]
            z = (np.maximum(np.einsum("nc,hc->nh", keys.astype(np.float64),
                                      q[r, 0].astype(np.float64)), 0) * w[r, 0]).sum(-1)
            order = np.lexsort((np.arange(N), -z))[:100]
            np.testing.assert_array_equal(out["topk"][r, 0], np.sort(order))


def test_mtp_step_scores_the_union_and_replays_the_accepted_rows(oracle_mod):
    """A whole speculative-decoding step (§3.2.2): the rows' selections (each with its own
    exploration draws) are unioned, every row is scored over the union, and the EMA replays
    rows 0..a of the accepted prefix: V = al^(a+1) V0 + (1-al) sum_r al^(a-r) z_r on every
    scored slot, the same closed form as the replay's own pin, applied to the step's scores."""
    o = oracle_mod
    rng = np.random.default_rng(33)
    R, H, d, n, rows = 2, 2, 8, 1200, 3
    kw = dict(n_req=R, max_slots=1280, max_rows=4, n_heads=H, head_dim=d, kv_heads=1,
              q_dtype="f32", k_dtype="f32", top_k=64, rho_bp=6000, gamma_bp=3000, alpha=0.9)
    cfg = o.make_cfg(**kw)
    MB = o.max_blocks(cfg)
    pool = rng.integers(-3, 4, (R * MB, 64, 1, d)).astype(np.float32)
    bt = np.arange(R * MB, dtype=np.int32).reshape(R, MB)
    V, D, warm = o.new_state(cfg)
    V[:] = rng.standard_normal(V.shape)
    D[:] = rng.standard_normal(D.shape)
    warm[:] = 1
    V0 = V.copy()
    q = rng.integers(-3, 4, (R, rows, H, d)).astype(np.float32)
    w = rng.integers(0, 3, (R, rows, H)).astype(np.float32)
    ns = np.array([n, n - 500], np.int32)
    acc = np.array([2, 1], np.int32)
    out = o.OracleStep(cfg).run(V, D, warm, q, w, pool, None, bt, ns, ns - 1, rows, 9, 2, accepted=acc)
    assert out["ok"]
    differ = False
    for r in range(R):
        sel = [set(out["blocks"][r, x, : out["n_blocks"][r, x]].tolist()) for x in range(rows)]
        scored = out["blist"][r, : out["n_list"][r]].tolist()
        assert scored == sorted(set().union(*sel))
        differ |= any(s != sel[0] for s in sel)
        a = int(acc[r])
        for k, blk in enumerate(scored):
            for s in range(64):
                i = blk * 64 + s
                if i >= ns[r]:
                    continue
                zs = [np.float64(out["scores"][r, x, k * 64 + s]) for x in range(a + 1)]
                want = 0.9 ** (a + 1) * np.float64(V0[r, i]) + 0.1 * sum(
                    0.9 ** (a - x) * zs[x] for x in range(a + 1))
                assert abs(V[r, i] - want) <= 1e-5 * (abs(want) + 1)
    assert differ  # the rows' own exploration draws make the union larger than row 0's selection


# ------------------------------------------------------------- pooling ablations (§4.6)

def _pool_inputs(oracle_mod, pooling, seed, n, combine="max", ints=True):
    cfg = tiny_cfg(oracle_mod, combine=combine, pooling=pooling)
    rng = np.random.default_rng(seed)
    if ints:  # small integers: every fp32 sum below is exact, whatever its order
        V = rng.integers(-50, 51, cfg.max_slots).astype(np.float32)
        D = rng.integers(-50, 51, oracle_mod.d_len(cfg)).astype(np.float32)
    else:
        V = rng.standard_normal(cfg.max_slots).astype(np.float32)
        D = rng.standard_normal(oracle_mod.d_len(cfg)).astype(np.float32)
    q = n + 3
    pred = np.maximum(V[:n], D[q - np.arange(n)]) if combine == "max" else V[:n] + D[q - np.arange(n)]
    return cfg, V, D, q, pred


@pytest.mark.parametrize("combine", ["max", "sum"])
@pytest.mark.parametrize("n", [1, 37, 64, 150, 257])
def test_mean_pooling_is_the_block_mean(oracle_mod, combine, n):
    """MEAN pooling: with integer predictions the fp32 sum is exact in any order, so the
    block score is the exact mean rounded once (numpy's float64 mean, then float32)."""
    cfg, V, D, q, pred = _pool_inputs(oracle_mod, "mean", 40 + n, n, combine)
    S = oracle_mod.block_scores(cfg, V, D, n, q)
    want = [np.float32(pred[j * 64: (j + 1) * 64].astype(np.float64).mean()) for j in range(-(-n // 64))]
    np.testing.assert_array_equal(S, np.array(want, np.float32))


@pytest.mark.parametrize("combine", ["max", "sum"])
@pytest.mark.parametrize("n", [1, 3, 64, 130, 257])
def test_top4_pooling_is_the_mean_of_the_four_largest(oracle_mod, combine, n):
    """TOP4 pooling: the mean of the four largest slot predictions of a block (all of them
    when the block has fewer), exact for integer predictions."""
    cfg, V, D, q, pred = _pool_inputs(oracle_mod, "top4", 70 + n, n, combine)
    S = oracle_mod.block_scores(cfg, V, D, n, q)
    want = []
    for j in range(-(-n // 64)):
        blk = np.sort(pred[j * 64: (j + 1) * 64].astype(np.float64))[::-1][:4]
        want.append(np.float32(blk.mean()))
    np.testing.assert_array_equal(S, np.array(want, np.float32))


@pytest.mark.parametrize("n", [64, 200])
def test_pooling_invariants_on_real_values(oracle_mod, n):
    """Non-integer predictions: max >= top-4 mean >= mean (up to rounding of the means), a
    constant block pools to its constant under every pooling, and a one-slot block to its
    only value."""
    cfgs = {p: tiny_cfg(oracle_mod, pooling=p) for p in ("max", "mean", "top4")}
    _, V, D, q, _ = _pool_inputs(oracle_mod, "max", 5, n, ints=False)
    S = {p: oracle_mod.block_scores(c, V, D, n, q) for p, c in cfgs.items()}
    eps = 1e-6
    assert np.all(S["max"] >= S["top4"] - eps * np.abs(S["max"]))
    assert np.all(S["top4"] >= S["mean"] - eps * np.abs(S["top4"]))
    Vc = np.full_like(V, np.float32(0.3))
    Dc = np.full_like(D, np.float32(-1.0))
    for p, c in cfgs.items():
        np.testing.assert_array_equal(oracle_mod.block_scores(c, Vc, Dc, n, q), np.float32(0.3))
    for p, c in cfgs.items():  # N = 65: the second block holds one slot
        S1 = oracle_mod.block_scores(c, V, D, 65, 68)
        assert S1[1] == max(V[64], D[68 - 64])


# ------------------------------------------------------- A0 block reduction (§4.6)

@pytest.mark.parametrize("combine", ["max", "sum"])
@pytest.mark.parametrize("n,top_k", [(290, 16), (150, 40), (64, 16), (297, 1)])
def test_a0_selects_the_blocks_of_the_top_k_predicted_slots(oracle_mod, combine, n, top_k):
    """A0: numpy brute force -- the K slots with the largest predicted score (ties: lower
    slot), then every block holding one, plus the sink and newest blocks."""
    o = oracle_mod
    cfg = tiny_cfg(o, combine=combine, pooling="slots", top_k=top_k, n_req=1, rho_bp=6000)
    rng = np.random.default_rng(n + top_k)
    V = rng.integers(-5, 6, cfg.max_slots).astype(np.float32)   # small integers: many ties
    D = rng.integers(-5, 6, o.d_len(cfg)).astype(np.float32)
    q = n + 2
    warm = np.ones(1, np.int32)
    blocks, nb_, _, _, ok = o.select_blocks(cfg, V[None], D[None], warm, np.array([n], np.int32),
                                            np.array([q], np.int32), 1, -1, 0, 0)
    assert ok
    i = np.arange(n)
    pred = np.maximum(V[:n], D[q - i]) if combine == "max" else V[:n] + D[q - i]
    order = np.lexsort((i, -pred.astype(np.float64)))
    nblk = -(-n // 64)
    want = sorted(set((order[:top_k] // 64).tolist()) | {0, nblk - 1})
    assert blocks[0, 0, : nb_[0, 0]].tolist() == want


def test_a0_dense_cases(oracle_mod):
    """Cold requests, budgets of every block (rho = 0) and K >= N select every block."""
    o = oracle_mod
    n = 280
    for rho, top_k, warm in ((4000, 16, 0), (0, 16, 1), (4000, 300, 1)):
        cfg = tiny_cfg(o, pooling="slots", top_k=top_k, n_req=1, rho_bp=rho)
        rng = np.random.default_rng(rho + top_k)
        V = rng.standard_normal(cfg.max_slots).astype(np.float32)
        D = rng.standard_normal(o.d_len(cfg)).astype(np.float32)
        blocks, nb_, _, _, ok = o.select_blocks(cfg, V[None], D[None], np.array([warm], np.int32),
                                                np.array([n], np.int32), np.array([n + 1], np.int32),
                                                1, -1, 0, 0)
        assert ok and blocks[0, 0, : nb_[0, 0]].tolist() == list(range(-(-n // 64)))


def test_a0_hand_example_each_top_slot_alone_in_its_block(oracle_mod):
    """A0 on predictions that put each of the K = 3 best slots in a block of its own, and
    every other prediction far below: dropping any one of the K slots would drop its block.
    A budget of every block (rho = 0) still selects every block."""
    o = oracle_mod
    n = 640                                                   # 10 blocks
    for rho, want in ((4000, [0, 2, 4, 6, 9]), (0, list(range(10)))):
        cfg = tiny_cfg(o, pooling="slots", top_k=3, n_req=1, rho_bp=rho, max_slots=n)
        V = np.full(cfg.max_slots, -100.0, np.float32)
        D = np.full(o.d_len(cfg), -100.0, np.float32)
        V[2 * 64 + 5], V[4 * 64 + 1], V[6 * 64 + 63] = 10.0, 9.0, 8.0
        V[6 * 64 + 62] = 7.0                                  # 4th best: same block as the 3rd
        V[8 * 64] = 6.0                                       # 5th best: a block of its own
        blocks, nb_, _, _, ok = o.select_blocks(cfg, V[None], D[None], np.ones(1, np.int32),
                                                np.array([n], np.int32), np.array([n - 1], np.int32),
                                                1, -1, 0, 0)
        assert ok and blocks[0, 0, : nb_[0, 0]].tolist() == want


# ------------------------------------------------------- A2 block reduction (§4.6)

def _a2_step(o, cfg, V, D, n, q, blocks, zfun):
    """Score the listed blocks with zfun(slot) and apply the oracle's A2 update (one row)."""
    MB = o.max_blocks(cfg)
    blist = np.full((1, MB), -1, np.int32)
    blist[0, : len(blocks)] = blocks
    scores = np.zeros((1, 1, MB * 64), np.float32)
    for k, b in enumerate(blocks):
        for s in range(64):
            scores[0, 0, k * 64 + s] = zfun(b * 64 + s)
    warm = np.zeros(1, np.int32)
    assert o.replay_ema(cfg, V, D, warm, scores, blist, np.array([len(blocks)], np.int32),
                        np.array([n], np.int32), np.array([q], np.int32), 1)
    return warm


def test_a2_update_closed_form(oracle_mod):
    """A2: n equal observations of a block give alpha^n V0 + (1 - alpha^n) z for the
    block-level V and for the diagonal entry at the block offset floor(q/64) - j; the
    observation is the block's max over its live slots; other entries stay unchanged."""
    o = oracle_mod
    cfg = tiny_cfg(o, pooling="a2", n_req=1, alpha=0.9)
    n, q = 200, 203                      # blocks 0..3, the last holding slots 192..199
    V = np.zeros((1, cfg.max_slots), np.float32)
    D = np.zeros((1, o.d_len(cfg)), np.float32)
    V[0, :4] = [1.0, -2.0, 0.5, 3.0]
    D[0, :4] = [0.25, -1.0, 2.0, 0.0]
    V0, D0 = V.copy(), D.copy()
    # slot values: block 1 peaks at slot 100 (7.0), block 3's live slots peak at 199 (-0.5);
    # slots past N (200..255) hold larger values, which must be ignored
    z = lambda i: {100: 7.0, 199: -0.5}.get(i, -0.5 if 192 <= i < 200 else (9.0 if i >= 200 else -3.0))
    for step in range(5):
        warm = _a2_step(o, cfg, V, D, n, q, [1, 3], z)
        assert warm[0] == 1
    qb = q // 64
    a5 = 0.9 ** 5
    for j, zb in ((1, 7.0), (3, -0.5)):
        assert abs(V[0, j] - (a5 * V0[0, j] + (1 - a5) * zb)) < 1e-5
        assert abs(D[0, qb - j] - (a5 * D0[0, qb - j] + (1 - a5) * zb)) < 1e-5
    assert V[0, 0] == V0[0, 0] and V[0, 2] == V0[0, 2]          # unscored blocks
    assert D[0, qb - 0] == D0[0, qb] and D[0, qb - 2] == D0[0, qb - 2]
    assert np.all(V[0, 4:] == 0) and np.all(D[0, 4:] == 0)      # no slot-level entries touched


@pytest.mark.parametrize("combine", ["max", "sum"])
def test_a2_selection_ranks_block_states(oracle_mod, combine):
    """A2 selection: with D = -inf-like (or 0 under sum) the top blocks are numpy's ranking
    of V's block entries; with V low the ranking follows D read at floor(q/64) - j, which
    pins the direction of the block offset."""
    o = oracle_mod
    n, q = 297, 300                       # 5 blocks, query block 4
    cfg = tiny_cfg(o, combine=combine, pooling="a2", n_req=1, rho_bp=4000, gamma_bp=0)
    rng = np.random.default_rng(3)
    nb = 5
    m = max(-(-cfg.top_k // 64), -(-(10000 - 4000) * nb // 10000))
    for which in ("V", "D"):
        V = np.full((1, cfg.max_slots), -1e6 if which == "D" else 0.0, np.float32)
        D = np.full((1, o.d_len(cfg)), -1e6 if which == "V" else 0.0, np.float32)
        if combine == "sum":
            (D if which == "V" else V)[:] = 0.0
        vals = rng.permutation(nb).astype(np.float32)
        if which == "V":
            V[0, :nb] = vals
            score = vals
        else:
            D[0, q // 64 - np.arange(nb)] = vals
            score = vals
        blocks, nbk, _, _, ok = o.select_blocks(cfg, V, D, np.ones(1, np.int32), np.array([n], np.int32),
                                                np.array([q], np.int32), 1, -1, 0, 0)
        assert ok
        free = [j for j in range(nb) if j not in (0, nb - 1)]
        ranked = sorted(free, key=lambda j: (-score[j], j))[: m - 2]
        assert blocks[0, 0, : nbk[0, 0]].tolist() == sorted({0, nb - 1} | set(ranked))


def test_a2_refuses_several_rows(oracle_mod):
    o = oracle_mod
    cfg = tiny_cfg(o, pooling="a2", n_req=1)
    V, D, warm = o.new_state(cfg)
    *_, ok = o.select_blocks(cfg, V, D, warm, np.array([200], np.int32), np.array([203], np.int32), 2)
    assert not ok


# ------------------------------------------------ block-age exploration (§4.6)

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_block_age_exploration_takes_the_least_recently_observed(oracle_mod, seed):
    """Block-age exploration: numpy brute force -- the forced blocks, the top m - f - e blocks
    by score (lower block on ties), then the e not yet selected blocks with the smallest age
    (the step + 1 of their last observation, 0 = never), lower block on equal ages."""
    o = oracle_mod
    n, q = 64 * 40 - 5, 64 * 40 - 2                  # 40 blocks
    cfg = tiny_cfg(o, explore="age", n_req=1, max_slots=64 * 40, rho_bp=5000, gamma_bp=2500, top_k=16)
    rng = np.random.default_rng(seed)
    V = rng.integers(-20, 21, (1, cfg.max_slots)).astype(np.float32)
    D = np.full((1, o.d_len(cfg)), -1e6, np.float32)
    age = rng.integers(0, 6, (1, o.max_blocks(cfg))).astype(np.uint32)   # many equal ages
    blocks, nbk, _, _, ok = o.select_blocks(cfg, V, D, np.ones(1, np.int32), np.array([n], np.int32),
                                            np.array([q], np.int32), 1, -1, 3, 0, age=age)
    assert ok
    nb = 40
    S = np.array([V[0, j * 64:min((j + 1) * 64, n)].max() for j in range(nb)])
    m = max(-(-16 // 64), -(-(10000 - 5000) * nb // 10000))
    f = 2
    e = min(2500 * m // 10000, m - f)
    free = [j for j in range(1, nb - 1)]
    top = sorted(free, key=lambda j: (-S[j], j))[: m - f - e]
    rest = [j for j in free if j not in top]
    explore = sorted(rest, key=lambda j: (int(age[0, j]), j))[:e]
    assert e > 0 and blocks[0, 0, : nbk[0, 0]].tolist() == sorted({0, nb - 1} | set(top) | set(explore))


def test_block_age_update_marks_the_listed_blocks(oracle_mod):
    o = oracle_mod
    cfg = tiny_cfg(o, explore="age", n_req=2)
    MB = o.max_blocks(cfg)
    age = np.full((2, MB), 7, np.uint32)
    blist = np.full((2, MB), -1, np.int32)
    blist[0, :3] = [0, 2, 4]
    blist[1, :1] = [1]
    assert o.block_age_update(cfg, age, blist, np.array([3, 1], np.int32), np.array([300, 100], np.int32), 41)
    want = np.full((2, MB), 7, np.uint32)
    want[0, [0, 2, 4]] = 42
    want[1, 1] = 42
    np.testing.assert_array_equal(age, want)
    blist[1, 0] = 3                                     # outside a 100-slot context
    assert not o.block_age_update(cfg, age, blist, np.array([3, 1], np.int32), np.array([300, 100], np.int32), 41)


def test_block_age_mode_needs_ages_and_one_row(oracle_mod):
    o = oracle_mod
    cfg = tiny_cfg(o, explore="age", n_req=1)
    V, D, warm = o.new_state(cfg)
    ns, qp = np.array([200], np.int32), np.array([203], np.int32)
    assert not o.select_blocks(cfg, V, D, warm, ns, qp)[-1]
    age = np.zeros((1, o.max_blocks(cfg)), np.uint32)
    assert o.select_blocks(cfg, V, D, warm, ns, qp, age=age)[-1]
    assert not o.select_blocks(cfg, V, D, warm, ns, qp, rows=2, age=age)[-1]
