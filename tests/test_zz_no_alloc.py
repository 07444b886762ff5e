"""The allocation-free selection entry point, spin_select_blocks_noalloc.

Some callers cannot allocate device memory for a workspace (engines that reserve all
device memory up front in their own pool, plugin hosts that give the library no
allocator, latency-critical loops that must not allocate).  For them the library offers
a variant of the block selection that uses a scratch array built into the library
instead of a caller workspace.  These tests call it through the C ABI and check that it
returns exactly what spin_select_blocks returns, on two calls in a row (the second call
reuses the array the first one left behind), and that oversized configurations are
refused.  This file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

from sparse_attention_indexer_spin_gb300 import spin
from sparse_attention_indexer_spin_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


def _warm_workload(wl):
    inp = syn.SyntheticInputs(wl, "cuda")
    cfg = spin.make_config(**wl.config_fields())
    st = spin.LayerState(cfg)
    spin.init_state(cfg, st.V, st.D, st.Vmax, st.warm)
    buf = spin.StepBuffers(cfg, wl.rows)
    for step in range(2):                     # a dense step, then a sparse one
        q, w, qp = inp.step_inputs()
        acc = torch.zeros(wl.n_req, dtype=torch.int32, device="cuda") if wl.rows > 1 else None
        spin.run_step(cfg, st, buf, q, w, inp.k_pool[0], inp.k_scale[0], inp.n_pages,
                      inp.block_table, inp.n_slots, qp, step, 0, None, acc)
        inp.advance(step, acc.cpu() if acc is not None else None)
    torch.cuda.synchronize()
    return inp, cfg, st, buf


@pytest.mark.parametrize("name,rows,n_req,n0", [("v4flash", 1, 6, 9000), ("mtp", 4, 6, 9000),
                                                 ("v4flash", 1, 1, 9000 * 64)])
def test_noalloc_select_equals_workspace_select(spin_lib, name, rows, n_req, n0):
    """The third case has more than 8192 blocks per request, so the selection runs the
    shared-memory kernel, which reads the scratch array at its largest offsets."""
    wl = syn.CONFIGS[name].replace(n_req=n_req, n0=n0, steps=4, n_heads=8, head_dim=64,
                                   q_dtype="f32", k_dtype="f32", kv_heads=8, top_k=256,
                                   rows=rows, mean_accept=2.4 if rows > 1 else 0.0)
    inp, cfg, st, buf = _warm_workload(wl)
    R, MB = cfg.n_req, cfg.max_blocks
    qp = (inp.n_slots - 1).to(torch.int32)
    for call, step in enumerate((7, 8)):      # two calls in a row
        ref_b = torch.full((R, rows, MB), -1, dtype=torch.int32, device="cuda")
        ref_n = torch.zeros((R, rows), dtype=torch.int32, device="cuda")
        ref_u = torch.full((R, MB), -1, dtype=torch.int32, device="cuda")
        ref_nu = torch.zeros((R,), dtype=torch.int32, device="cuda")
        got_b, got_n = ref_b.clone(), ref_n.clone()
        got_u, got_nu = ref_u.clone(), ref_nu.clone()
        status = torch.zeros((1,), dtype=torch.int32, device="cuda")
        spin.select_blocks(cfg, st.V, st.D, st.Vmax, st.warm, inp.n_slots, qp, rows, None, step,
                           0, ref_b, ref_n, ref_u if rows > 1 else None,
                           ref_nu if rows > 1 else None, buf.workspace, status)
        spin.select_blocks_noalloc(cfg, st.V, st.D, st.Vmax, st.warm, inp.n_slots, qp, rows, None,
                                   step, 0, got_b, got_n, got_u if rows > 1 else None,
                                   got_nu if rows > 1 else None, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(got_n, ref_n), call
        assert torch.equal(got_b, ref_b), call
        if rows > 1:
            assert torch.equal(got_nu, ref_nu) and torch.equal(got_u, ref_u), call
        # the selection is sparse: the comparison is not between two dense lists
        nb = -(-inp.n_slots.long() // 64)
        assert bool((ref_n[:, 0].long() < nb).all())


def test_noalloc_rejects_oversized_configuration(spin_lib):
    # 96 requests x 4 rows x 4112 blocks needs 1.58 M scratch entries, above the 1 M built in
    wl = syn.CONFIGS["mtp"].replace(n_req=96)
    cfg = spin.make_config(**wl.config_fields())
    rc = spin.lib().spin_select_blocks_noalloc(ctypes.byref(cfg), *([None] * 6), 4, None, 0, 0,
                                               *([None] * 6))
    assert rc == 3
    assert "scratch" in spin.lib().spin_last_error_string().decode()
