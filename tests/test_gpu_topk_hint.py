"""GPU parity of the temporal (hinted) top-K against the CPU oracle's top-K.

The hinted top-K must return exactly what the plain top-K returns, whatever its hint says:
the hint only decides which path computes it.  Two groups of tests:

- direct: the hint's records and candidate arrays are written on the host from the scores
  (the live slots whose order key is at or above a chosen guess, in shuffled order), so that
  each branch of the kernel is reached on purpose -- a hit, ties at the guess, a miss (fewer
  than K candidates), an overflow (more than cap), no guess, fewer live slots than K, and a
  boundary bin too large for the candidate array;
- end to end: decode steps through the C ABI with the score kernels (streaming, tcgen05 bf16
  and e4m3, several verifier rows, generic) collecting the candidates, teacher-forced
  against the oracle step by step, with most steps resolved from the candidates.
"""
import numpy as np
import pytest
import torch

from _parity import Harness, np_
from oracle import oracle as o
from sparse_attention_indexer_spin_gb300 import spin
from sparse_attention_indexer_spin_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

W = spin.HINT_WORDS
GUESS, COUNT, EXTRA, HIT, MISS, OVER, COLD, EXACT, LAST, FLAGS = range(10)


@pytest.fixture(scope="module", autouse=True)
def _lib(spin_lib):
    assert torch.cuda.is_available(), "these tests need a GPU"
    return spin_lib


def _fields(n_req, max_slots, rows, top_k):
    return dict(n_req=n_req, max_slots=max_slots, max_rows=rows, n_heads=8, head_dim=64, kv_heads=8,
                q_dtype="f32", k_dtype="f32", top_k=top_k, rho_bp=4000, gamma_bp=500, alpha=0.9)


def order_keys(z):
    """The order-preserving uint32 image of float32 scores (larger float, larger key; -0 as +0)."""
    u = np.ascontiguousarray(z, np.float32).view(np.uint32).copy()
    u[(u & 0x7FFFFFFF) == 0] = 0
    neg = (u & 0x80000000) != 0
    return np.where(neg, ~u, u | 0x80000000).astype(np.uint32)


def key_float(k):
    """The float32 of an order key (inverse of order_keys)."""
    k = np.uint32(k)
    bits = k & np.uint32(0x7FFFFFFF) if k & np.uint32(0x80000000) else ~k
    return float(np.array([bits], np.uint32).view(np.float32)[0])


def live_positions(blist, n_list, n_slots, r):
    lst = blist[r, : n_list[r]].astype(np.int64)
    slot = (lst[:, None] * 64 + np.arange(64)[None, :]).ravel()
    return np.nonzero(slot < n_slots[r])[0]


def plant(hint, cfg, rows, scores, blist, n_list, n_slots, guess_rank, rng, extra=0, collected=True):
    """Write each row's record and candidates as a score kernel with this guess would: the
    threshold is the key at `guess_rank` (None: no guess), the candidates every live slot at or
    above it, in random order.  collected=False writes only the guess (the threshold over the
    weights' sum, exact for a sum of 4) and leaves the collection to the top-K kernel.
    Returns the counts."""
    R, cap = cfg.n_req, _cap(cfg)
    recs = np.zeros((R * rows, W), np.uint32)
    cands = np.zeros((R * rows, cap), np.uint64)
    counts = []
    for r in range(R):
        pos = live_positions(blist, n_list, n_slots, r)
        for row in range(rows):
            rr = r * rows + row
            keys = order_keys(scores[r, row, pos])
            if guess_rank is None or len(keys) == 0:
                counts.append(0)
                recs[rr, EXTRA] = extra
                continue
            g = np.sort(keys)[::-1][min(guess_rank, len(keys)) - 1]
            take = keys >= g
            ent = (keys[take].astype(np.uint64) << np.uint64(32)) | (~pos[take].astype(np.uint32)).astype(np.uint64)
            rng.shuffle(ent)
            c = len(ent)
            counts.append(c)
            recs[rr, EXTRA] = extra
            if collected:
                cands[rr, : min(c, cap)] = ent[:cap]
                recs[rr, GUESS], recs[rr, COUNT], recs[rr, FLAGS] = g, c, 1
            else:
                recs[rr, GUESS] = order_keys(np.array([key_float(g) / WSUM], np.float32))[0]
    raw = hint.buf
    rec_bytes = (R * rows * W * 4 + 255) // 256 * 256
    raw[: recs.nbytes].copy_(torch.from_numpy(recs.view(np.uint8).ravel()))
    raw[rec_bytes: rec_bytes + cands.nbytes].copy_(torch.from_numpy(cands.view(np.uint8).ravel()))
    return counts


def _cap(cfg):
    """The library's candidate capacity for these shapes (8 K, at least 4096; all fit)."""
    c = 4096
    while c < 8 * cfg.top_k:
        c *= 2
    return c


WSUM = 4.0  # the direct tests' head weights: 8 heads of 0.5


def run_hinted(cfg, rows, scores, blist, n_list, n_slots, hint):
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = torch.full((cfg.n_req, rows, cfg.top_k), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    w = torch.full((cfg.n_req, rows, cfg.n_heads), WSUM / cfg.n_heads, dtype=torch.float32, device="cuda")
    spin.topk_hinted(cfg, d(scores), w, d(blist), d(n_list), d(n_slots), rows, out, hint, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out.cpu().numpy()


# (n_req, max_slots, rows, top_k, dist, guess rank as a multiple of K (None: no guess), branch)
CASES = [
    pytest.param(3, 131072, 1, 2048, "normal", 1.5, HIT, id="hit"),
    pytest.param(3, 131072, 1, 2048, "ties", 1.2, None, id="ties-at-guess"),
    pytest.param(2, 131072, 1, 2048, "narrow", 1.5, HIT, id="hit-narrow"),
    pytest.param(3, 131072, 1, 2048, "normal", 0.5, MISS, id="miss"),
    pytest.param(3, 131072, 1, 512, "normal", 10.0, OVER, id="overflow"),
    pytest.param(3, 131072, 1, 2048, "normal", None, COLD, id="cold"),
    pytest.param(2, 131072, 1, 1024, "ties", None, None, id="cold-ties"),
    pytest.param(2, 131072, 1, 512, "narrow", None, COLD, id="cold-narrow-refined"),
    pytest.param(4, 4000, 1, 2048, "normal", None, COLD, id="fewer-than-K"),
    pytest.param(2, 65536, 1, 512, "equal", None, EXACT, id="equal-exact"),
    pytest.param(2, 65536, 4, 1024, "normal", 1.7, HIT, id="4rows"),
    pytest.param(40, 65536, 1, 512, "normal", 2.0, HIT, id="many-rows"),
    pytest.param(3, 262144, 1, 256, "normal", 1.3, HIT, id="small-K-long-list"),
]


@pytest.mark.parametrize("collected", [True, False], ids=["score-collected", "self-collected"])
@pytest.mark.parametrize("n_req,max_slots,rows,top_k,dist,mult,branch", CASES)
def test_topk_hinted_direct(n_req, max_slots, rows, top_k, dist, mult, branch, collected):
    f = _fields(n_req, max_slots, rows, top_k)
    cfg, ocfg = spin.make_config(**f), o.make_cfg(**f)
    scores, blist, n_list, n_slots = syn.topk_inputs(n_req, max_slots, rows, dist, 100 + n_req)
    want, ok = o.topk(ocfg, scores, blist, n_list, n_slots, rows)
    assert ok
    hint = spin.TopkHint(cfg, rows)
    rng = np.random.default_rng(7)
    rank = None if mult is None else max(1, int(mult * top_k))
    counts = plant(hint, cfg, rows, scores, blist, n_list, n_slots, rank, rng, collected=collected)
    got = run_hinted(cfg, rows, scores, blist, n_list, n_slots, hint)
    np.testing.assert_array_equal(got, want)
    rec = hint.records()
    assert (rec[:, COUNT] == 0).all() and (rec[:, FLAGS] == 0).all()   # consumed
    assert (rec[:, LAST] == np.array(counts, np.uint32)).all()
    if branch is not None:
        col = EXACT if branch == EXACT else branch
        assert (rec[:, col] == 1).all(), rec[:, HIT:LAST]
        if branch != EXACT:   # a boundary bin that fits after refinement needs no exact passes
            assert (rec[:, EXACT] == 0).all(), rec[:, HIT:LAST]
    # a next guess (0: none), times the weights' sum, admits at least K live slots of these scores
    for r in range(n_req):
        pos = live_positions(blist, n_list, n_slots, r)
        for row in range(rows):
            g = int(rec[r * rows + row, GUESS])
            if g:
                thr = np.float32(key_float(g)) * np.float32(WSUM)
                assert (scores[r, row, pos] >= thr).sum() >= min(len(pos), top_k)


def test_topk_hinted_margin_adapts():
    """A miss doubles the rank margin, an overflow halves it, within [K/8, cap/2 - K]."""
    f = _fields(1, 131072, 1, 1024)
    cfg = spin.make_config(**f)
    scores, blist, n_list, n_slots = syn.topk_inputs(1, 131072, 1, "normal", 5)
    hint = spin.TopkHint(cfg, 1)
    rng = np.random.default_rng(1)
    plant(hint, cfg, 1, scores, blist, n_list, n_slots, 512, rng, extra=300)      # miss
    run_hinted(cfg, 1, scores, blist, n_list, n_slots, hint)
    assert int(hint.records()[0, EXTRA]) == 600
    plant(hint, cfg, 1, scores, blist, n_list, n_slots, 9000, rng, extra=600)     # overflow (cap 8192)
    run_hinted(cfg, 1, scores, blist, n_list, n_slots, hint)
    assert int(hint.records()[0, EXTRA]) == 300
    plant(hint, cfg, 1, scores, blist, n_list, n_slots, 512, rng, extra=2000)     # miss at the top
    run_hinted(cfg, 1, scores, blist, n_list, n_slots, hint)
    assert int(hint.records()[0, EXTRA]) == 8192 // 2 - 1024


def test_topk_hinted_reset_and_errors():
    f = _fields(3, 131072, 1, 2048)
    cfg = spin.make_config(**f)
    hint = spin.TopkHint(cfg, 1)
    hint.buf.fill_(0xAB)
    hint.reset(req=1)
    rec = hint.records()
    assert (rec[1] == 0).all() and (rec[0] != 0).all() and (rec[2] != 0).all()
    hint.reset()
    assert (hint.records() == 0).all()
    big = spin.make_config(**_fields(1, 131072, 1, 4096))             # K above 2048
    with pytest.raises(spin.SpinError) as e:
        spin.topk_hint_size(big, 1)
    assert e.value.code == 4


# ----------------------------------------------------------------------- end to end

def run_hinted_steps(h, steps, hint, score_requests=None):
    inp = h.inp
    for step in range(steps):
        q, w, qp = inp.step_inputs()
        acc = inp.draw_accepted().cuda() if h.wl.rows > 1 else None
        h.step(step, 0, q, w, qp, accepted=acc, score_requests=score_requests, hint=hint)
        inp.advance(step, acc)
    return hint.stats()


def _tc_workload(k_dtype, rows, n_req=3, n0=6000, seed=31):
    return syn.Workload("tc", n_req=n_req, n_layers=1, n0=n0, n_heads=64, head_dim=128,
                        kv_heads=1, q_dtype="bf16", k_dtype=k_dtype, top_k=256, rho_bp=4000,
                        gamma_bp=500, alpha=0.9, steps=8, rows=rows, heavy=8, rope_dims=64,
                        shuffle=True, mean_accept=2.0 if rows > 1 else 0.0, seed=seed)


@pytest.mark.parametrize("path", ["stream", "generic"])
def test_hinted_pr1_all_steps(path):
    """The 4096-slot, 8-head fp32 workload, every one of its 32 steps, with the streaming and
    the generic score kernel collecting the candidates."""
    h = Harness(syn.CONFIGS["pr1"], score_path=path)
    hint = spin.TopkHint(h.cfg, 1)
    st = run_hinted_steps(h, h.wl.steps, hint)
    assert st["cold"] == 1 and st["hit"] >= 24, st


@pytest.mark.parametrize("k_dtype,rows", [("bf16", 1), ("e4m3", 1), ("bf16", 4), ("e4m3", 2)])
def test_hinted_tcgen05(k_dtype, rows):
    h = Harness(_tc_workload(k_dtype, rows), score_path="tcgen05")
    hint = spin.TopkHint(h.cfg, rows)
    st = run_hinted_steps(h, 8, hint)
    assert st["hit"] >= 5 * h.wl.n_req * rows, st


def test_hinted_reset_request_goes_cold():
    """After a request's state and hint are reset, its next step is dense and cold."""
    h = Harness(syn.CONFIGS["pr1"].replace(n_req=3, steps=6))
    hint = spin.TopkHint(h.cfg, 1)
    run_hinted_steps(h, 3, hint)
    st = h.states[0]
    spin.init_state(h.cfg, st.V, st.D, st.Vmax, st.warm, 1)
    hint.reset(req=1)
    before = hint.records()[:, COLD].copy()
    q, w, qp = h.inp.step_inputs()
    h.step(3, 0, q, w, qp, hint=hint)
    after = hint.records()[:, COLD]
    assert (after - before).tolist() == [0, 1, 0]


def test_hinted_v32_full_size():
    """131072 slots, 64 heads x 128, a bf16 key per head, K = 2048: 6 steps of one layer."""
    h = Harness(syn.CONFIGS["v32"], layers=1)
    hint = spin.TopkHint(h.cfg, 1)
    st = run_hinted_steps(h, 6, hint, score_requests=[0])
    assert st["hit"] >= 4, st


def test_hinted_serving_full_size():
    h = Harness(syn.CONFIGS["serving"])
    hint = spin.TopkHint(h.cfg, 1)
    st = run_hinted_steps(h, 5, hint, score_requests=[0, 95])
    assert st["hit"] >= 300, st


def test_hinted_mtp_full_size():
    h = Harness(syn.CONFIGS["mtp"])
    hint = spin.TopkHint(h.cfg, 4)
    st = run_hinted_steps(h, 4, hint, score_requests=[0])
    assert st["hit"] >= 2 * 16 * 4, st
