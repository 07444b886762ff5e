"""A whole decode step -- selection (with the decode step read from device memory), score,
top-K and EMA update of every layer -- captured once in a CUDA graph and replayed for the
following steps gives bit-identical states and outputs to the eager calls."""
import pytest
import torch

from sparse_attention_indexer_spin_gb300 import spin
from sparse_attention_indexer_spin_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(spin_lib):
    assert torch.cuda.is_available(), "these tests need a GPU"
    return spin_lib


def _same(a_states, b_states, a_buf, b_buf):
    for sa, sb in zip(a_states, b_states):
        for n in ("V", "D", "Vmax", "warm"):
            assert torch.equal(getattr(sa, n), getattr(sb, n)), n
    for n in ("blocks", "n_blocks", "scores", "topk", "status"):
        assert torch.equal(getattr(a_buf, n), getattr(b_buf, n)), n


@pytest.mark.parametrize("name,over", [
    ("pr1", dict(n_req=3, n0=3000, n_layers=2, steps=6)),
    ("v4flash", dict(n_req=4, n0=20000, n_layers=2, steps=6)),
])
def test_graph_replay_equals_eager(name, over):
    wl = syn.CONFIGS[name].replace(**over)
    inp = syn.SyntheticInputs(wl, "cuda")
    cfg = spin.make_config(**wl.config_fields())
    L = inp.n_layers
    eager = [spin.LayerState(cfg) for _ in range(L)]
    graphed = [spin.LayerState(cfg) for _ in range(L)]
    for st in eager + graphed:
        spin.init_state(cfg, st.V, st.D, st.Vmax, st.warm)
    buf_e, buf_g = spin.StepBuffers(cfg), spin.StepBuffers(cfg)
    q, w, qp = inp.step_inputs()
    q_s, w_s, qp_s = q.clone(), w.clone(), qp.clone()          # the graph's static inputs
    step_dev = torch.zeros(1, dtype=torch.int64, device="cuda")

    def graph_step():
        for l in range(L):
            spin.run_step(cfg, graphed[l], buf_g, q_s, w_s, inp.k_pool[l], inp.k_scale[l], inp.n_pages,
                          inp.block_table, inp.n_slots, qp_s, step_dev, l)

    # step 0 runs uncaptured on both sides (first calls do their one-time host setup)
    for l in range(L):
        spin.run_step(cfg, eager[l], buf_e, q, w, inp.k_pool[l], inp.k_scale[l], inp.n_pages,
                      inp.block_table, inp.n_slots, qp, 0, l)
    graph_step()
    torch.cuda.synchronize()
    _same(eager, graphed, buf_e, buf_g)
    inp.advance(0)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        graph_step()
    for step in range(1, wl.steps):
        q, w, qp = inp.step_inputs()
        for l in range(L):
            spin.run_step(cfg, eager[l], buf_e, q, w, inp.k_pool[l], inp.k_scale[l], inp.n_pages,
                          inp.block_table, inp.n_slots, qp, step, l)
        q_s.copy_(q)
        w_s.copy_(w)
        qp_s.copy_(qp)
        step_dev.fill_(step)
        g.replay()
        torch.cuda.synchronize()
        _same(eager, graphed, buf_e, buf_g)
        assert int(buf_g.status.item()) == 0
        inp.advance(step)
