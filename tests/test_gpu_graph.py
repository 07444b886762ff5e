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


@pytest.mark.parametrize("name,over,topk", [
    ("v4flash", dict(n_req=4, n0=20000, n_layers=2), "hinted"),
    ("v32", dict(n_req=1, n0=6000, n_layers=3), "hinted"),
    ("mtp", dict(n_req=3, n0=8000, n_layers=2), "plain"),
])
def test_bench_graph_step_equals_eager(name, over, topk):
    """The bench's captured layer-stacked step (selection with a device step for every layer,
    each layer's score and top-K -- temporal or plain -- then one EMA or MTP commit launch),
    replayed step after step, gives the eager steps' states and outputs bit for bit."""
    import bench
    base = syn.CONFIGS[name].replace(**over)
    eager = bench.Workload(base, 8, base.rho_bp, topk=topk, schedule="stacked")
    graphed = bench.Workload(base, 8, base.rho_bp, share=eager, topk=topk, schedule="stacked")
    for s in range(2):
        eager.step(s)
        graphed.step(s)
    graphed.capture_graph()
    for s in range(2, 8):
        eager.step(s)
        graphed.replay_steps([s])
        for n in ("V", "D", "Vmax", "warm"):
            assert torch.equal(getattr(eager.state, n), getattr(graphed.state, n)), (s, n)
        assert torch.equal(eager.scores, graphed.scores) and torch.equal(eager.topk, graphed.topk), s
        assert torch.equal(eager.n_blocks[s], graphed.n_blocks[0]), s
        if base.rows > 1:
            assert torch.equal(eager.n_unions[s], graphed.n_unions[0]), s
    assert int(graphed.buf.status.item()) == 0 and int(eager.buf.status.item()) == 0
