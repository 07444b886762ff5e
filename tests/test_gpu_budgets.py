"""Per-layer block budgets on the GPU (sparse_attention_indexer_spin_gb300.budgets): the dense
probe's top-K against the oracle's top-K of the probe's scores over every block, each layer's
miss curve against the oracle's curve from the oracle's own block predictions, the device
table against the allocation, and every budgeted step's selection size against the table."""
import numpy as np
import pytest
import torch

from oracle import budgets as ob
from oracle import oracle as o
from sparse_attention_indexer_spin_gb300 import spin
from sparse_attention_indexer_spin_gb300 import synthetic as syn
from sparse_attention_indexer_spin_gb300.budgets import BudgetController

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(spin_lib):
    assert torch.cuda.is_available(), "these tests need a GPU"
    return spin_lib


def test_probe_curves_table_and_budgeted_steps():
    L, P, steps, n_points = 3, 4, 10, 101
    wl = syn.CONFIGS["pr1"].replace(n_req=4, n0=6000, n_layers=L, steps=steps, shuffle=True)
    inp = syn.SyntheticInputs(wl, "cuda")
    cfg, ocfg = spin.make_config(**wl.config_fields()), o.make_cfg(**wl.config_fields())
    R, MB, K = cfg.n_req, cfg.max_blocks, cfg.top_k
    ctl = BudgetController(cfg, L, target_rho_bp=4000, period=P, n_points=n_points)
    states = [spin.LayerState(cfg) for _ in range(L)]
    for st in states:
        spin.init_state(cfg, st.V, st.D, st.Vmax, st.warm)
    buf = spin.StepBuffers(cfg)
    probed_real = False
    for step in range(steps):
        q, w, qp = inp.step_inputs()
        ns = inp.n_slots.cpu().numpy().copy()
        qpn = qp.cpu().numpy().copy()
        nb = (ns.astype(np.int64) + 63) // 64
        for layer in range(L):
            st = states[layer]
            V, D = st.V.cpu().numpy().copy(), st.D.cpu().numpy().copy()
            warm = st.warm.cpu().numpy().copy()
            rho = int(ctl.table[layer].item())
            buf.status.zero_()
            ctl.step(st, buf, q, w, inp.k_pool[layer], inp.k_scale[layer], inp.n_pages, inp.block_table,
                     inp.n_slots, qp, step, layer)
            torch.cuda.synchronize()
            assert int(buf.status.item()) == 0
            n_blocks = buf.n_blocks[:, 0].cpu().numpy()
            if ctl.is_probe(step):
                assert n_blocks.tolist() == nb.tolist()  # the probe scores every block
                blist = np.full((R, MB), -1, np.int32)
                for r in range(R):
                    blist[r, : nb[r]] = np.arange(nb[r])
                want_topk, ok = o.topk(ocfg, buf.scores.cpu().numpy(), blist, nb.astype(np.int32), ns, 1)
                assert ok
                topk = buf.topk[:, 0, :].cpu().numpy()
                np.testing.assert_array_equal(topk, want_topk[:, 0, :])
                S = [o.block_scores(ocfg, V[r], D[r], int(ns[r]), int(qpn[r])).tolist() for r in range(R)]
                tk = [topk[r].tolist() if warm[r] else [-1] * K for r in range(R)]
                want = ob.mean_miss_curve(S, nb.tolist(), tk, K, n_points)
                np.testing.assert_array_equal(ctl.curves[layer], np.array(want, np.float32))
                probed_real |= bool(warm.any()) and max(want) > 0
            else:
                for r in range(R):
                    m = o.budget(int(nb[r]), K, rho)
                    dense = (not warm[r]) or nb[r] <= 2 or m >= nb[r]
                    assert n_blocks[r] == (nb[r] if dense else max(m, 2)), (step, layer, r, rho)
        if ctl.is_probe(step):
            ctl.publish()
            torch.cuda.synchronize()
            g, rho_all = spin.allocate_budgets(ctl.curves, ctl.target_g)
            assert ctl.table.cpu().numpy().tolist() == rho_all.tolist()
            assert int(g.sum()) == L * ctl.target_g
        inp.advance(step)
    assert probed_real  # a probe on warm requests measured a non-zero curve
