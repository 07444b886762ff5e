"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle.

Block masks, union lists and top-K indices must be bit-exact; V, D and Vmax bit-exact;
scores within 1e-3 (fp32/bf16 inputs) or 2e-2 (FP8 keys) of the magnitude bound.
"""
import numpy as np
import pytest
import torch

from _parity import Harness, np_
from oracle import oracle as o
from sparse_attention_indexer_spin_gb300 import spin
from sparse_attention_indexer_spin_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(spin_lib):
    assert torch.cuda.is_available(), "these tests need a GPU"
    return spin_lib


def run_steps(h, steps, layer=0, check_every=1, score_requests=None, rho=None):
    inp = h.inp
    out = None
    for step in range(steps):
        q, w, qp = inp.step_inputs()
        acc = inp.draw_accepted().cuda() if h.wl.rows > 1 else None
        out = h.step(step, layer, q, w, qp, rho_override=rho, accepted=acc,
                     check=(step % check_every == 0), score_requests=score_requests)
        inp.advance(step, acc)
    return out


# ------------------------------------------------------------------ small workloads

def test_pr1_teacher_forced_all_steps():
    """The 1-request, 4096-slot, 8-head fp32 workload: every one of its 32 steps."""
    h = Harness(syn.CONFIGS["pr1"])
    out = run_steps(h, h.wl.steps)
    assert out["worst"] < 1e-3


@pytest.mark.parametrize("path", ["generic", "stream"])
def test_pr1_score_paths(path):
    h = Harness(syn.CONFIGS["pr1"].replace(steps=4), score_path=path)
    run_steps(h, 4)


@pytest.mark.parametrize("combine,alpha", [("sum", 0.9), ("max", 0.5)])
def test_combiner_and_alpha(combine, alpha):
    wl = syn.CONFIGS["pr1"].replace(combine=combine, alpha=alpha, steps=6, n_req=3, n0=3001,
                                    gamma_bp=2000)
    h = Harness(wl)
    run_steps(h, 6)


def test_ragged_requests_tiny_heads():
    """Several requests of ragged lengths, a shared key and tiny heads (generic kernel)."""
    wl = syn.Workload("tiny", n_req=5, n_layers=1, n0=700, n_heads=2, head_dim=4, kv_heads=1,
                      q_dtype="f32", k_dtype="f32", top_k=40, rho_bp=5000, gamma_bp=2000,
                      alpha=0.9, steps=8, heavy=3, rope_dims=2, shuffle=True, seed=11)
    h = Harness(wl)
    h.inp.n_slots.copy_(torch.tensor([700, 1, 64, 65, 0], dtype=torch.int32))
    run_steps(h, 8)


@pytest.mark.parametrize("n_req,n0,top_k", [(2, 1500, 128), (32, 1500, 128), (2, 40000, 2048)])
def test_integer_inputs_free_running_bit_exact(n_req, n0, top_k):
    """Integer-valued q, k, w make every score exact: the GPU and the oracle run free
    (each on its own state) and must agree bit for bit at every step.  Integer scores tie
    often, so the K-th score is usually shared (cut in slot order); the longer context
    takes the top-K's sampled bracket, and 32 requests the one-CTA-per-row top-K."""
    wl = syn.Workload("int", n_req=n_req, n_layers=1, n0=n0, n_heads=8, head_dim=64, kv_heads=8,
                      q_dtype="f32", k_dtype="f32", top_k=top_k, rho_bp=4000, gamma_bp=1000,
                      alpha=0.9, steps=10, heavy=0, rope_dims=0, seed=5)
    h = Harness(wl)
    g = torch.Generator(device="cuda").manual_seed(9)
    for p in h.inp.k_pool:
        p.copy_(torch.randint(-3, 4, p.shape, generator=g, device="cuda").float())
    ocfg = h.ocfg
    V, D, warm = o.new_state(ocfg)
    pool = np_(h.inp.k_pool[0])
    bt = np_(h.inp.block_table)
    st = h.states[0]
    for step in range(wl.steps):
        q = torch.randint(-2, 3, (n_req, 1, 8, 64), generator=g, device="cuda").float()
        w = torch.randint(0, 3, (n_req, 1, 8), generator=g, device="cuda").float()
        qp = (h.inp.n_slots - 1).clamp_min(0).to(torch.int32)
        h.buf.status.zero_()
        spin.run_step(h.cfg, st, h.buf, q, w, h.inp.k_pool[0], None, h.inp.n_pages,
                      h.inp.block_table, h.inp.n_slots, qp, step, 0)
        res = o.OracleStep(ocfg).run(V, D, warm, np_(q), np_(w), pool, None, bt,
                                     np_(h.inp.n_slots), np_(qp), 1, step, 0)
        torch.cuda.synchronize()
        gnb = np_(h.buf.n_blocks)
        np.testing.assert_array_equal(gnb, res["n_blocks"])
        np.testing.assert_array_equal(np_(h.buf.topk), res["topk"])
        assert np_(st.V).tobytes() == V.tobytes()
        assert np_(st.D).tobytes() == D.tobytes()
        h.inp.advance(step)


def test_rho_zero_is_dense_and_equals_dense_topk():
    wl = syn.CONFIGS["pr1"].replace(rho_bp=0, steps=3, n_req=2)
    h = Harness(wl)
    out = run_steps(h, 3)
    nb = -(-np_(h.inp.n_slots) // 64)
    np.testing.assert_array_equal(out["n_blocks"][:, 0], nb)


def test_rho_override_device_table():
    wl = syn.CONFIGS["pr1"].replace(steps=4, n_req=2)
    h = Harness(wl)
    rho = torch.tensor([6500], dtype=torch.int32, device="cuda")
    run_steps(h, 4, rho=rho)


def test_long_context_selection_fallback():
    """More than 8192 blocks per request: selection takes the shared-memory kernel instead of
    the register-resident one (and top-K the single-CTA kernel)."""
    wl = syn.Workload("long", n_req=2, n_layers=1, n0=530000, n_heads=2, head_dim=16, kv_heads=1,
                      q_dtype="f32", k_dtype="bf16", top_k=256, rho_bp=4000, gamma_bp=500,
                      alpha=0.9, steps=3, heavy=4, rope_dims=8, seed=3)
    assert wl.max_blocks > 8192
    h = Harness(wl)
    run_steps(h, 3)


def test_eight_verifier_rows():
    """The largest row count (one 8-CTA cluster per request in the selection)."""
    wl = syn.CONFIGS["mtp"].replace(n_req=2, n0=5000, steps=3, n_heads=8, head_dim=64, rows=8,
                                    mean_accept=3.0)
    h = Harness(wl)
    run_steps(h, 3)


# --------------------------------------------------------------- tensor-core kernel

def _tc_workload(k_dtype, rows, n_req=3, n0=2000, seed=21):
    return syn.Workload("tc", n_req=n_req, n_layers=1, n0=n0, n_heads=64, head_dim=128,
                        kv_heads=1, q_dtype="bf16", k_dtype=k_dtype, top_k=256, rho_bp=4000,
                        gamma_bp=500, alpha=0.9, steps=4, rows=rows, heavy=8, rope_dims=64,
                        shuffle=True, mean_accept=2.0 if rows > 1 else 0.0, seed=seed)


@pytest.mark.parametrize("k_dtype,rows", [("bf16", 1), ("e4m3", 1), ("bf16", 4), ("e4m3", 2),
                                          ("bf16", 3), ("e4m3", 3), ("e4m3", 4)])
def test_tcgen05_small_ragged(k_dtype, rows):
    """Shared key, 64 heads x 128 dims: requests of 2000, 130 and 64 slots (odd block lists
    leave half-empty 128-slot tiles), through the tcgen05 kernel."""
    h = Harness(_tc_workload(k_dtype, rows), score_path="tcgen05")
    h.inp.n_slots.copy_(torch.tensor([2000, 130, 64], dtype=torch.int32))
    run_steps(h, 4)


def test_tcgen05_negative_fp8_scales():
    """FP8 per-slot scales of either sign: the scale multiplies the dot product before the
    ReLU, so a negative scale selects the negative dot products."""
    h = Harness(_tc_workload("e4m3", 1, seed=23), score_path="tcgen05")
    g = torch.Generator(device="cuda").manual_seed(3)
    sc = h.inp.k_scale[0]
    flip = torch.rand(sc.shape, generator=g, device="cuda") < 0.3
    sc[flip] = -sc[flip]
    run_steps(h, 3)


@pytest.mark.parametrize("k_dtype", ["bf16", "e4m3"])
def test_tcgen05_matches_generic_kernel(k_dtype):
    """Independent GPU cross-check: the tensor-core and the generic CUDA-core kernel on
    the same selection."""
    wl = _tc_workload(k_dtype, 1, n_req=4, n0=5000, seed=3)
    h = Harness(wl, score_path="tcgen05")
    q, w, qp = h.inp.step_inputs()
    h.step(0, 0, q, w, qp)
    cfg_g = spin.make_config(**wl.config_fields(), score_path="generic")
    out = torch.zeros_like(h.buf.scores)
    spin.indexer_score(cfg_g, q, w, h.inp.k_pool[0], h.inp.k_scale[0], h.inp.n_pages,
                       h.inp.block_table, h.buf.blocks, h.buf.n_blocks, h.inp.n_slots, 1, out,
                       h.buf.status)
    torch.cuda.synchronize()
    nb = h.buf.n_blocks[:, 0].tolist()
    for r in range(wl.n_req):
        a, b = out[r, 0, : nb[r] * 64], h.buf.scores[r, 0, : nb[r] * 64]
        assert torch.allclose(a, b, rtol=1e-4, atol=1e-3), (r, (a - b).abs().max())


# ------------------------------------------------------------------------- top-K paths

def test_topk_many_rows_ragged():
    """40 requests (enough rows for the one-CTA-per-row top-K) of ragged lengths."""
    wl = syn.CONFIGS["pr1"].replace(n_req=40, n0=6000, steps=3, gamma_bp=1000, shuffle=True)
    h = Harness(wl)
    ns = torch.randint(1, 6000, (40,), generator=torch.Generator().manual_seed(4)).to(torch.int32)
    h.inp.n_slots.copy_(ns)
    run_steps(h, 3)


def test_topk_all_equal_scores():
    """Degenerate case: w = 0 makes every score 0, so the top-K is the K lowest slot ids
    (and the boundary bin overflows the collection buffer of the per-row kernel)."""
    wl = syn.CONFIGS["v4flash"].replace(n_req=36, n0=20000, steps=2, n_heads=8, head_dim=64,
                                        kv_heads=8, q_dtype="f32", k_dtype="f32", top_k=512)
    h = Harness(wl)
    for step in range(2):
        q, w, qp = h.inp.step_inputs()
        out = h.step(step, 0, q, torch.zeros_like(w), qp)
        h.inp.advance(step)
    for r in range(wl.n_req):
        blks = out["blist"][r, : out["nlist"][r]]
        ids = (blks[:, None] * 64 + np.arange(64)[None, :]).ravel()
        ids = ids[ids < np_(h.inp.n_slots)[r]]
        np.testing.assert_array_equal(out["topk"][r, 0], np.sort(ids)[: wl.top_k])


# ------------------------------------------------------------------------------- MTP

def test_mtp_small_union_and_replay():
    wl = syn.CONFIGS["mtp"].replace(n_req=3, n0=3000, steps=6, n_heads=8, head_dim=64,
                                    q_dtype="f32", k_dtype="f32", top_k=256)
    h = Harness(wl)
    out = run_steps(h, 6)
    assert (out["nlist"] >= out["n_blocks"][:, 0]).all()


def test_commit_a0_equals_update():
    """accepted = 0 for every request: the MTP commit equals the one-row update of row 0."""
    wl = syn.CONFIGS["mtp"].replace(n_req=2, n0=2000, steps=2, n_heads=8, head_dim=64,
                                    q_dtype="f32", k_dtype="f32", top_k=128)
    h = Harness(wl)
    q, w, qp = h.inp.step_inputs()
    acc = torch.zeros(2, dtype=torch.int32, device="cuda")
    h.step(0, 0, q, w, qp, accepted=acc)
    st = h.states[0]
    V0, D0 = st.V.clone(), st.D.clone()
    q, w, qp = h.inp.step_inputs()
    h.step(1, 0, q, w, qp, accepted=None, check=False)        # scores only, no commit
    Va, Da = st.V.clone(), st.D.clone()
    assert torch.equal(Va, V0)
    spin.commit_mtp(h.cfg, st.V, st.D, st.Vmax, st.warm, h.buf.scores, 4, h.buf.union,
                    h.buf.n_union, h.inp.n_slots, qp, acc, h.buf.status)
    Vc, Dc = st.V.clone(), st.D.clone()
    st.V.copy_(Va); st.D.copy_(Da)
    row0 = h.buf.scores.new_zeros((2, 1, h.cfg.max_blocks * 64))
    row0[:, 0] = h.buf.scores[:, 0]
    spin.update_ema(h.cfg, st.V, st.D, st.Vmax, st.warm, row0, h.buf.union, h.buf.n_union,
                    h.inp.n_slots, qp, h.buf.status)
    torch.cuda.synchronize()
    assert torch.equal(st.V, Vc) and torch.equal(st.D, Dc)


# ------------------------------------------------------------------------- edge cases

def test_status_bits_and_skips():
    wl = syn.CONFIGS["pr1"].replace(n_req=3, steps=2)
    h = Harness(wl)
    q, w, qp = h.inp.step_inputs()
    h.step(0, 0, q, w, qp)                                     # warm everything up
    st, buf, cfg = h.states[0], h.buf, h.cfg
    # bad q for request 1: its selection is empty and the status says so
    qp_bad = qp.clone()
    qp_bad[1] = 5
    buf.status.zero_()
    spin.select_blocks(cfg, st.V, st.D, st.Vmax, st.warm, h.inp.n_slots, qp_bad, 1, None, 1, 0,
                       buf.blocks, buf.n_blocks, None, None, buf.workspace, buf.status)
    torch.cuda.synchronize()
    assert int(buf.status.item()) & spin.STATUS_BITS["BAD_QPOS"]
    assert int(buf.n_blocks[1, 0].item()) == 0 and int(buf.n_blocks[0, 0].item()) > 0
    # bad page id: its block scores 0 and BAD_PAGE is raised
    bt = h.inp.block_table.clone()
    blk0 = int(buf.blocks[0, 0, 0].item())
    bt[0, blk0] = h.inp.n_pages + 7
    buf.status.zero_()
    spin.indexer_score(cfg, q, w, h.inp.k_pool[0], None, h.inp.n_pages, bt, buf.blocks,
                       buf.n_blocks, h.inp.n_slots, 1, buf.scores, buf.status)
    torch.cuda.synchronize()
    assert int(buf.status.item()) & spin.STATUS_BITS["BAD_PAGE"]
    assert float(buf.scores[0, 0, :64].abs().sum().item()) == 0.0
    # accepted out of range: state untouched
    V0 = st.V.clone()
    acc = torch.tensor([0, 3, 0], dtype=torch.int32, device="cuda")
    buf.status.zero_()
    spin.commit_mtp(cfg, st.V, st.D, st.Vmax, st.warm, buf.scores, 1, buf.blocks, buf.n_blocks,
                    h.inp.n_slots, qp, acc, buf.status)
    torch.cuda.synchronize()
    assert int(buf.status.item()) & spin.STATUS_BITS["BAD_ACCEPTED"]
    assert torch.equal(st.V[1], V0[1])


def test_host_validation_errors():
    cfg = spin.make_config(**syn.CONFIGS["pr1"].config_fields())
    bad = spin.make_config(**{**syn.CONFIGS["pr1"].config_fields(), "block": 32})
    st = spin.LayerState(cfg)
    with pytest.raises(spin.SpinError) as e:
        spin.init_state(bad, st.V, st.D, st.Vmax, st.warm)
    assert e.value.code == 1
    buf = spin.StepBuffers(cfg)
    with pytest.raises(spin.SpinError):  # rows > max_rows
        spin.topk(cfg, buf.scores, buf.blocks, buf.n_blocks, st.warm, 2, buf.topk, buf.status)


def test_topk_pads_with_minus_one():
    wl = syn.CONFIGS["pr1"].replace(n_req=1, n0=100, top_k=256, steps=1)
    h = Harness(wl)
    out = run_steps(h, 1)
    assert (out["topk"][0, 0, 100:] == -1).all()
    np.testing.assert_array_equal(out["topk"][0, 0, :100], np.arange(100))


def test_reset_one_request():
    wl = syn.CONFIGS["pr1"].replace(n_req=2, steps=2)
    h = Harness(wl)
    run_steps(h, 2)
    st = h.states[0]
    V1 = st.V[1].clone()
    spin.init_state(h.cfg, st.V, st.D, st.Vmax, st.warm, 0)
    torch.cuda.synchronize()
    assert float(st.V[0].abs().sum()) == 0 and int(st.warm[0]) == 0 and int(st.warm[1]) == 1
    assert torch.equal(st.V[1], V1)


# -------------------------------------------------------------- full-size workloads

def test_v32_full_size_one_layer():
    """131072 slots, 64 heads x 128 dims, a bf16 key per head, K = 2048: 3 steps of one
    layer, every score of every step checked."""
    h = Harness(syn.CONFIGS["v32"], layers=1)
    out = run_steps(h, 3)
    assert out["worst"] < 1e-3


def test_v4flash_full_size_sampled():
    """32 requests x 131072 slots, FP8 keys with a per-slot scale, shuffled pages: a dense
    first step and four sparse ones; selection, top-K and EMA checked for every request,
    scores for two requests."""
    h = Harness(syn.CONFIGS["v4flash"])
    run_steps(h, 5, score_requests=[0, 31])


def test_serving_full_size_sampled():
    """96 requests x 131072 slots, FP8 keys: a dense first step and four sparse ones."""
    h = Harness(syn.CONFIGS["serving"])
    run_steps(h, 5, score_requests=[0, 95])


def test_mtp_full_size_sampled():
    """16 requests x 262144 slots, 4 verifier rows: a dense first step and four sparse ones
    with their unions and deferred commits."""
    h = Harness(syn.CONFIGS["mtp"])
    run_steps(h, 5, score_requests=[0])


# ------------------------------------------------------------------ pooling ablations

@pytest.mark.parametrize("pooling", ["mean", "top4", "slots", "a2"])
@pytest.mark.parametrize("combine", ["max", "sum"])
def test_pooling_ablations(pooling, combine):
    """The block-reduction ablations of §4.6 (A1 with mean or top-4 pooling; A0, the top-K
    predicted slots expanded to their blocks; A2, block-level EMAs of max-pooled scores):
    selections and EMA states bit-identical to the oracle's on ragged contexts (one of them
    all forced blocks), every step teacher-forced."""
    wl = syn.CONFIGS["pr1"].replace(pooling=pooling, combine=combine, steps=6, n_req=3, n0=3001,
                                    gamma_bp=1000)
    h = Harness(wl)
    h.inp.n_slots.copy_(torch.tensor([3001, 700, 65], dtype=torch.int32))
    run_steps(h, 6)


@pytest.mark.parametrize("pooling", ["top4", "slots"])
def test_pooling_ablation_many_rows(pooling):
    """Top-4 pooling and A0 with four verifier rows (per-row selections and their union);
    top-4 runs the 16-blocks-per-warp instance."""
    wl = syn.CONFIGS["mtp"].replace(pooling=pooling, n_req=3, n0=5000, steps=4, n_heads=8, head_dim=64,
                                    q_dtype="f32", k_dtype="f32", top_k=256)
    h = Harness(wl)
    run_steps(h, 4)


def test_a0_many_requests_and_budget_table():
    """A0 over 40 requests (the sampled top-K kernel's instance), with a sparsity read from a
    device table and then a table of 0 (every block)."""
    wl = syn.CONFIGS["pr1"].replace(pooling="slots", n_req=40, n0=2500, steps=4, top_k=128)
    h = Harness(wl)
    run_steps(h, 2, rho=torch.tensor([5000], dtype=torch.int32, device="cuda"))
    run_steps(h, 2, rho=torch.tensor([0], dtype=torch.int32, device="cuda"))


def test_a2_refuses_several_rows():
    """A2 keeps block-level state for one query row: several rows are refused on the host."""
    wl = syn.CONFIGS["pr1"].replace(pooling="a2", n_req=2, rows=2, mean_accept=1.5)
    cfg = spin.make_config(**wl.config_fields())
    st = spin.LayerState(cfg)
    buf = spin.StepBuffers(cfg)
    ns = torch.tensor([700, 300], dtype=torch.int32, device="cuda")
    blocks = torch.zeros((2, 2, cfg.max_blocks), dtype=torch.int32, device="cuda")
    nbk = torch.zeros((2, 2), dtype=torch.int32, device="cuda")
    un = torch.zeros((2, cfg.max_blocks), dtype=torch.int32, device="cuda")
    nun = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(spin.SpinError):
        spin.select_blocks(cfg, st.V, st.D, st.Vmax, st.warm, ns, ns - 1, 2, None, 0, 0, blocks, nbk, un, nun,
                           buf.workspace, buf.status)


# ------------------------------------------------------------------ block-age exploration

@pytest.mark.parametrize("combine", ["max", "sum"])
def test_block_age_exploration(combine):
    """Block-age exploration (§4.6, Staleness mitigation): selections bit-identical to the
    oracle's given the same ages, and the ages after each step equal to the oracle's update
    (listed blocks get step + 1), every step teacher-forced on ragged contexts."""
    wl = syn.CONFIGS["pr1"].replace(explore="age", combine=combine, steps=8, n_req=3, n0=3001, gamma_bp=2500)
    h = Harness(wl)
    h.inp.n_slots.copy_(torch.tensor([3001, 700, 65], dtype=torch.int32))
    run_steps(h, 8)
    assert int(h.ages[0].max().item()) == 8        # blocks scored at the last step


def test_block_age_entry_points():
    """Block-age exploration needs the age entry points and one row; the age entry points need
    the mode."""
    wl = syn.CONFIGS["pr1"].replace(explore="age", n_req=2)
    cfg = spin.make_config(**wl.config_fields())
    st, buf = spin.LayerState(cfg), spin.StepBuffers(cfg)
    ns = torch.tensor([700, 300], dtype=torch.int32, device="cuda")
    age = torch.zeros((2, cfg.max_blocks), dtype=torch.int32, device="cuda")
    with pytest.raises(spin.SpinError):
        spin.select_blocks(cfg, st.V, st.D, st.Vmax, st.warm, ns, ns - 1, 1, None, 0, 0, buf.blocks, buf.n_blocks,
                           None, None, buf.workspace, buf.status)
    with pytest.raises(spin.SpinError):
        spin.select_blocks_noalloc(cfg, st.V, st.D, st.Vmax, st.warm, ns, ns - 1, 1, None, 0, 0, buf.blocks,
                                   buf.n_blocks, None, None, buf.status)
    with pytest.raises(spin.SpinError):
        spin.update_ema(cfg, st.V, st.D, st.Vmax, st.warm, buf.scores, buf.blist, buf.n_list, ns, ns - 1,
                        buf.status)
    spin.select_blocks_age(cfg, st.V, st.D, st.Vmax, st.warm, ns, ns - 1, 1, None, 0, 0, age, buf.blocks,
                           buf.n_blocks, None, None, buf.workspace, buf.status)
    torch.cuda.synchronize()
    plain = spin.make_config(**syn.CONFIGS["pr1"].replace(n_req=2).config_fields())
    with pytest.raises(spin.SpinError):
        spin.select_blocks_age(plain, st.V, st.D, st.Vmax, st.warm, ns, ns - 1, 1, None, 0, 0, age, buf.blocks,
                               buf.n_blocks, None, None, buf.workspace, buf.status)


@pytest.mark.parametrize("pooling,explore", [("max", "random"), ("mean", "random"), ("top4", "random"),
                                             ("slots", "random"), ("a2", "random"), ("max", "age")])
def test_ablations_tiny_contexts(pooling, explore):
    """Empty, one-slot, one-block, one-block-plus-one and two-block contexts next to a long one,
    under the method and every ablation: selections, scores, top-K and state as the oracle's."""
    wl = syn.CONFIGS["pr1"].replace(pooling=pooling, explore=explore, n_req=6, n0=3001, steps=4,
                                    gamma_bp=2500)
    h = Harness(wl)
    h.inp.n_slots.copy_(torch.tensor([0, 1, 64, 65, 130, 3001], dtype=torch.int32))
    run_steps(h, 4)
