"""GPU tests of the layer-stacked calls (spin_select_blocks_layers, spin_update_ema_layers,
spin_commit_mtp_layers) through the C ABI.

A stacked call on arrays [L][...] must produce exactly what L single-layer calls on the
slices produce (the single-layer calls are themselves checked against the oracle in the
parity tests): the selections, unions and counts bit for bit, V, D, Vmax and warm bit for bit.
Each layer's state is first driven to a different, warm point by a few decode steps, so the
layers' selections differ.
"""
import numpy as np
import pytest
import torch

from _parity import np_
from oracle import oracle as o
from sparse_attention_indexer_spin_gb300 import spin
from sparse_attention_indexer_spin_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(spin_lib):
    assert torch.cuda.is_available(), "these tests need a GPU"
    return spin_lib


class Stack:
    """L layers' states stacked [L][...], warmed by a few single-layer decode steps each."""

    def __init__(self, wl, L, warm_steps=3):
        self.wl, self.L = wl, L
        self.inp = syn.SyntheticInputs(wl.replace(n_layers=L), "cuda")
        self.cfg = spin.make_config(**wl.config_fields())
        c, R, rows = self.cfg, wl.n_req, wl.rows
        self.V = torch.zeros((L, R, c.max_slots), dtype=torch.float32, device="cuda")
        self.D = torch.zeros((L, R, c.d_len), dtype=torch.float32, device="cuda")
        self.Vmax = torch.zeros((L, R, c.max_blocks), dtype=torch.float32, device="cuda")
        self.warm = torch.zeros((L, R), dtype=torch.int32, device="cuda")
        self.buf = spin.StepBuffers(c, rows)
        for layer in range(L):
            st = self.layer_state(layer)
            spin.init_state(c, st.V, st.D, st.Vmax, st.warm)
        for step in range(warm_steps):
            for layer in range(L):
                q, w, qp = self.inp.step_inputs()
                acc = self.inp.draw_accepted().cuda() if rows > 1 else None
                spin.run_step(c, self.layer_state(layer), self.buf, q, w, self.inp.k_pool[layer],
                              self.inp.k_scale[layer], self.inp.n_pages, self.inp.block_table,
                              self.inp.n_slots, qp, step, layer, None, acc)
            self.inp.advance(step, acc if rows > 1 else None)
        torch.cuda.synchronize()

    def layer_state(self, layer):
        st = spin.LayerState.__new__(spin.LayerState)
        st.V, st.D, st.Vmax, st.warm = self.V[layer], self.D[layer], self.Vmax[layer], self.warm[layer]
        return st

    def snapshot(self):
        return [t.clone() for t in (self.V, self.D, self.Vmax, self.warm)]

    def restore(self, snap):
        for t, s in zip((self.V, self.D, self.Vmax, self.warm), snap):
            t.copy_(s)


def _select_both(sk, rho_table, step, layer0=2):
    c, L, R, rows, MB = sk.cfg, sk.L, sk.wl.n_req, sk.wl.rows, sk.cfg.max_blocks
    qp = (sk.inp.n_slots - 1).to(torch.int32)
    ws1 = spin.workspace_size(c, rows)
    ws = torch.zeros(L * ws1 // 4 + 64, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got_b = torch.full((L, R, rows, MB), -1, dtype=torch.int32, device="cuda")
    got_n = torch.zeros((L, R, rows), dtype=torch.int32, device="cuda")
    got_u = torch.full((L, R, MB), -1, dtype=torch.int32, device="cuda")
    got_nu = torch.zeros((L, R), dtype=torch.int32, device="cuda")
    spin.select_blocks_layers(c, L, layer0, sk.V, sk.D, sk.Vmax, sk.warm, sk.inp.n_slots, qp, rows,
                              rho_table, step, got_b, got_n, got_u, got_nu, ws, status)
    ref_b, ref_n, ref_u, ref_nu = got_b.clone().fill_(-1), got_n.clone().zero_(), got_u.clone().fill_(-1), got_nu.clone().zero_()
    for layer in range(L):
        st = sk.layer_state(layer)
        rho = None if rho_table is None else rho_table[layer:layer + 1]
        spin.select_blocks(c, st.V, st.D, st.Vmax, st.warm, sk.inp.n_slots, qp, rows, rho, step,
                           layer0 + layer, ref_b[layer], ref_n[layer], ref_u[layer], ref_nu[layer],
                           sk.buf.workspace, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(got_n, ref_n) and torch.equal(got_nu, ref_nu)
    assert torch.equal(got_b, ref_b) and torch.equal(got_u, ref_u)
    return got_b, got_n, got_u, got_nu


@pytest.mark.parametrize("name,L,rows,n_req,n0,table", [
    ("pr1", 3, 1, 2, 6000, False),          # register-resident selection, one row
    ("pr1", 4, 1, 3, 6000, True),           # a per-layer sparsity table
    ("mtp", 2, 4, 3, 5000, False),          # four verifier rows: cluster union
    ("pr1", 2, 1, 1, 9000 * 64, False),     # more than 8192 blocks: the shared-memory kernel
])
def test_select_layers_equals_per_layer(name, L, rows, n_req, n0, table):
    wl = syn.CONFIGS[name].replace(n_req=n_req, n0=n0, steps=6, n_heads=8, head_dim=64, kv_heads=8,
                                   q_dtype="f32", k_dtype="f32", top_k=256, rows=rows,
                                   mean_accept=2.4 if rows > 1 else 0.0, gamma_bp=1000)
    sk = Stack(wl, L, warm_steps=2)
    rho = torch.tensor([1000 * (l + 2) for l in range(L)], dtype=torch.int32, device="cuda") if table else None
    b, nb, _, _ = _select_both(sk, rho, step=11)
    # the layers' states differ, and so do their selections
    assert any(not torch.equal(b[0], b[l]) for l in range(1, L))


def test_update_ema_layers_equals_per_layer():
    wl = syn.CONFIGS["pr1"].replace(n_req=3, n0=7000, steps=6, gamma_bp=1000)
    L = 3
    sk = Stack(wl, L)
    c, R, MB = sk.cfg, wl.n_req, sk.cfg.max_blocks
    b, nb, _, _ = _select_both(sk, None, step=9)
    qp = (sk.inp.n_slots - 1).to(torch.int32)
    g = torch.Generator(device="cuda").manual_seed(5)
    scores = torch.randn((L, R, 1, MB * 64), generator=g, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lst, nl = b[:, :, 0, :].contiguous(), nb[:, :, 0].contiguous()
    snap = sk.snapshot()
    spin.update_ema_layers(c, L, sk.V, sk.D, sk.Vmax, sk.warm, scores, lst, nl, sk.inp.n_slots, qp, status)
    got = sk.snapshot()
    sk.restore(snap)
    for layer in range(L):
        st = sk.layer_state(layer)
        spin.update_ema(c, st.V, st.D, st.Vmax, st.warm, scores[layer], lst[layer], nl[layer],
                        sk.inp.n_slots, qp, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for a, r in zip(got, sk.snapshot()):
        assert torch.equal(a, r)
    assert not torch.equal(got[0], snap[0])


def test_commit_mtp_layers_equals_per_layer():
    wl = syn.CONFIGS["mtp"].replace(n_req=3, n0=5000, steps=6, n_heads=8, head_dim=64,
                                    q_dtype="f32", k_dtype="f32", top_k=256)
    L, rows = 2, 4
    sk = Stack(wl, L)
    c, R, MB = sk.cfg, wl.n_req, sk.cfg.max_blocks
    _, _, u, nu = _select_both(sk, None, step=7)
    qp = (sk.inp.n_slots - 1).to(torch.int32)
    g = torch.Generator(device="cuda").manual_seed(6)
    scores = torch.randn((L, R, rows, MB * 64), generator=g, device="cuda")
    acc = torch.tensor([0, 3, 1], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    snap = sk.snapshot()
    spin.commit_mtp_layers(c, L, sk.V, sk.D, sk.Vmax, sk.warm, scores, rows, u, nu, sk.inp.n_slots, qp,
                           acc, status)
    got = sk.snapshot()
    sk.restore(snap)
    for layer in range(L):
        st = sk.layer_state(layer)
        spin.commit_mtp(c, st.V, st.D, st.Vmax, st.warm, scores[layer], rows, u[layer], nu[layer],
                        sk.inp.n_slots, qp, acc, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for a, r in zip(got, sk.snapshot()):
        assert torch.equal(a, r)


def test_select_layers_against_oracle():
    """The stacked selection of layer l equals the oracle's selection for layer layer0 + l."""
    wl = syn.CONFIGS["pr1"].replace(n_req=2, n0=6000, steps=6, gamma_bp=1500)
    sk = Stack(wl, 3)
    ocfg = o.make_cfg(**wl.config_fields())
    b, nb, _, _ = _select_both(sk, None, step=13, layer0=5)
    ns, qp = np_(sk.inp.n_slots), np_(sk.inp.n_slots) - 1
    for layer in range(3):
        ob, onb, _, _, ok = o.select_blocks(ocfg, np_(sk.V[layer]).copy(), np_(sk.D[layer]).copy(),
                                           np_(sk.warm[layer]).copy(), ns, qp.astype(np.int32), 1, -1, 13,
                                           5 + layer)
        assert ok
        np.testing.assert_array_equal(np_(nb[layer]), onb)
        for r in range(wl.n_req):
            np.testing.assert_array_equal(np_(b[layer])[r, 0, : onb[r, 0]], ob[r, 0, : onb[r, 0]])


def test_layers_host_validation():
    cfg = spin.make_config(**syn.CONFIGS["pr1"].config_fields())
    st = spin.LayerState(cfg)
    buf = spin.StepBuffers(cfg)
    with pytest.raises(spin.SpinError):           # workspace for one layer only
        spin.select_blocks_layers(cfg, 2, 0, st.V, st.D, st.Vmax, st.warm, st.warm, st.warm, 1, None, 0,
                                  buf.blocks, buf.n_blocks, None, None, buf.workspace, buf.status)
    with pytest.raises(spin.SpinError):           # no layers
        spin.update_ema_layers(cfg, 0, st.V, st.D, st.Vmax, st.warm, buf.scores, buf.blocks, buf.n_blocks,
                               st.warm, st.warm, buf.status)


@pytest.mark.parametrize("pooling,rows", [("slots", 1), ("slots", 4), ("a2", 1)])
def test_select_layers_ablations_equal_per_layer(pooling, rows):
    """A0 (the top-K predicted slots expanded to blocks) and A2 (block-level states) through
    the stacked call, with a per-layer sparsity table: identical to the per-layer calls."""
    base = syn.CONFIGS["pr1"] if rows == 1 else syn.CONFIGS["mtp"]
    wl = base.replace(pooling=pooling, n_req=2, n0=6000, steps=6, n_heads=8, head_dim=64, kv_heads=8,
                      q_dtype="f32", k_dtype="f32", top_k=256, rows=rows,
                      mean_accept=2.4 if rows > 1 else 0.0, gamma_bp=1000)
    L = 3
    sk = Stack(wl, L, warm_steps=2)
    rho = torch.tensor([3000, 5000, 7000], dtype=torch.int32, device="cuda")
    _select_both(sk, rho, step=4)
