"""Guard bands: every buffer the library writes is embedded in a larger allocation whose
margins hold a sentinel pattern.  After each step the margins must be intact, and the guarded
run must give bit-identical results to a run on plain buffers (the kernels are deterministic),
so no kernel writes outside its buffers or depends on what lies next to them.
"""
import pytest
import torch

from sparse_attention_indexer_spin_gb300 import spin
from sparse_attention_indexer_spin_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

GUARD = 4096                # elements on each side
SENTINEL = 0x7FBADBAD       # an int32 pattern (a NaN as fp32)


@pytest.fixture(scope="module", autouse=True)
def _lib(spin_lib):
    assert torch.cuda.is_available(), "these tests need a GPU"
    return spin_lib


class Guarded:
    """Replaces the 4-byte tensors of `obj` by views into guarded allocations."""

    def __init__(self, obj, names):
        self.big = {}
        for n in names:
            t = getattr(obj, n)
            assert t.element_size() == 4
            big = torch.empty(t.numel() + 2 * GUARD, dtype=t.dtype, device=t.device)
            big.view(torch.int32).fill_(SENTINEL)
            view = big[GUARD:GUARD + t.numel()].view(t.shape)
            view.copy_(t)
            setattr(obj, n, view)
            self.big[n] = big

    def check(self):
        for n, big in self.big.items():
            bits = big.view(torch.int32)
            assert bool((bits[:GUARD] == SENTINEL).all()), f"{n}: front band written"
            assert bool((bits[-GUARD:] == SENTINEL).all()), f"{n}: back band written"


STATE = ("V", "D", "Vmax", "warm")
BUFS = ("blocks", "n_blocks", "union", "n_union", "scores", "topk", "workspace", "status")


@pytest.mark.parametrize("name,over", [
    ("pr1", dict(n_req=3, n0=3000, steps=4)),
    ("v4flash", dict(n_req=4, n0=20000, steps=4)),
    ("v32", dict(n_req=1, n0=8192, steps=4, n_layers=1)),
    ("mtp", dict(n_req=3, n0=6000, steps=4)),
])
def test_guard_bands_and_identical_results(name, over):
    wl = syn.CONFIGS[name].replace(**over)
    inp = syn.SyntheticInputs(wl, "cuda", layers=1)
    cfg = spin.make_config(**wl.config_fields())
    plain_st, guard_st = spin.LayerState(cfg), spin.LayerState(cfg)
    for st in (plain_st, guard_st):
        spin.init_state(cfg, st.V, st.D, st.Vmax, st.warm)
    plain_buf, guard_buf = spin.StepBuffers(cfg, wl.rows), spin.StepBuffers(cfg, wl.rows)
    gs, gb = Guarded(guard_st, STATE), Guarded(guard_buf, BUFS)
    for step in range(wl.steps):
        q, w, qp = inp.step_inputs()
        acc = inp.draw_accepted().cuda() if wl.rows > 1 else None
        for st, buf in ((plain_st, plain_buf), (guard_st, guard_buf)):
            spin.run_step(cfg, st, buf, q, w, inp.k_pool[0], inp.k_scale[0], inp.n_pages,
                          inp.block_table, inp.n_slots, qp, step, 0, None, acc)
        torch.cuda.synchronize()
        gs.check()
        gb.check()
        assert int(guard_buf.status.item()) == 0
        for n in STATE:
            assert torch.equal(getattr(plain_st, n), getattr(guard_st, n)), (step, n)
        for n in ("blocks", "n_blocks", "topk", "scores"):
            assert torch.equal(getattr(plain_buf, n), getattr(guard_buf, n)), (step, n)
        inp.advance(step, acc)
