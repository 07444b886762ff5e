"""Free-running GPU-vs-oracle parity with integer-valued inputs, and FP8 query ranges.

Integer-valued q, k and w (exact in bf16, in e4m3 with a unit scale, and in fp32) make every
score exact and independent of the summation order, so the GPU and the oracle can each run
free on their own state for many steps and must still agree bit for bit on every output:
block lists, MTP unions, top-K indices (integer scores tie often, so the K-th score is
usually shared and cut by slot order), V, D and the warm flags.  One case per score kernel
and key format the workloads use: the per-head streaming kernel with bf16 keys (the
DeepSeek-V3.2-like shape) and with e4m3 keys, the tcgen05 kernel with a shared bf16 and a
shared e4m3 key, and the 4-row speculative-decoding loop with its deferred commit; the
one-row cases run with the plain and with the temporal top-K.

The FP8 query split (two e4m3 terms per element) is checked on rows whose elements span a
wide range -- one large element and the rest several orders of magnitude smaller -- against
the 2e-2 relative bound of the magnitude A_i.
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


def _integer_pools(h, g):
    """Replace the key pools by integers in [-3, 3] (e4m3 codes of them with unit scales)."""
    for layer, p in enumerate(h.inp.k_pool):
        vals = torch.randint(-3, 4, p.shape, generator=g, device="cuda")
        if h.wl.k_dtype == "e4m3":
            p.copy_(vals.float().to(torch.float8_e4m3fn).view(torch.uint8))
            h.inp.k_scale[layer].fill_(1.0)
        else:
            p.copy_(vals.to(p.dtype))


def _free_running(wl, score_path, steps, hinted=False, seed=9):
    h = Harness(wl, score_path=score_path)
    g = torch.Generator(device="cuda").manual_seed(seed)
    _integer_pools(h, g)
    R, rows, H, d = wl.n_req, wl.rows, wl.n_heads, wl.head_dim
    ocfg = h.ocfg
    V, D, warm = o.new_state(ocfg)
    pool = np_(h.inp.k_pool[0])
    scale = None if h.inp.k_scale[0] is None else np_(h.inp.k_scale[0])
    bt = np_(h.inp.block_table)
    st, buf = h.states[0], h.buf
    hint = spin.TopkHint(h.cfg, rows) if hinted else None
    qdt = syn.TORCH_DTYPE[wl.q_dtype]
    for step in range(steps):
        q = torch.randint(-2, 3, (R, rows, H, d), generator=g, device="cuda").to(qdt)
        w = torch.randint(0, 3, (R, rows, H), generator=g, device="cuda").float()
        qp = (h.inp.n_slots - 1).clamp_min(0).to(torch.int32)
        acc = h.inp.draw_accepted().cuda() if rows > 1 else None
        buf.status.zero_()
        spin.run_step(h.cfg, st, buf, q, w, h.inp.k_pool[0], h.inp.k_scale[0], h.inp.n_pages,
                      h.inp.block_table, h.inp.n_slots, qp, step, 0, None, acc, hint=hint)
        res = o.OracleStep(ocfg).run(V, D, warm, np_(q), np_(w), pool, scale, bt, np_(h.inp.n_slots),
                                     np_(qp), rows, step, 0, accepted=None if acc is None else np_(acc))
        torch.cuda.synchronize()
        assert res["ok"]
        assert int(buf.status.item()) == 0, "status %#x" % int(buf.status.item())
        gnb, gb = np_(buf.n_blocks), np_(buf.blocks)
        np.testing.assert_array_equal(gnb, res["n_blocks"])
        for r in range(R):
            for k in range(rows):
                np.testing.assert_array_equal(gb[r, k, : gnb[r, k]], res["blocks"][r, k, : gnb[r, k]])
        if rows > 1:
            gnu, gu = np_(buf.n_union), np_(buf.union)
            np.testing.assert_array_equal(gnu, res["n_union"])
            for r in range(R):
                np.testing.assert_array_equal(gu[r, : gnu[r]], res["union"][r, : gnu[r]])
        np.testing.assert_array_equal(np_(buf.topk), res["topk"])
        assert np_(st.V).tobytes() == V.tobytes(), "V differs at step %d" % step
        assert np_(st.D).tobytes() == D.tobytes(), "D differs at step %d" % step
        np.testing.assert_array_equal(np_(st.warm), warm)
        h.inp.advance(step, acc)
    return hint


def _wl(name, **kw):
    return syn.Workload(name, **{**dict(n_layers=1, n_heads=64, head_dim=128, q_dtype="bf16", rho_bp=4000,
                                        gamma_bp=1000, alpha=0.9, steps=8, heavy=0, rope_dims=0, seed=13),
                                 **kw})


@pytest.mark.parametrize("hinted", [False, True], ids=["plain-topk", "temporal-topk"])
def test_free_running_v32_stream_bf16(hinted):
    """A bf16 key per head (the DeepSeek-V3.2-like shape): the streaming kernel."""
    wl = _wl("v32int", n_req=2, n0=20000, kv_heads=64, k_dtype="bf16", top_k=2048)
    hint = _free_running(wl, "stream", 7, hinted)
    if hint is not None:
        assert hint.stats()["hit"] >= 4


def test_free_running_stream_e4m3_per_head():
    """An e4m3 key per head with its per-slot scale: the streaming kernel's FP8 instance."""
    wl = _wl("e4m3ph", n_req=2, n0=9000, kv_heads=64, k_dtype="e4m3", top_k=512)
    _free_running(wl, "stream", 6)


@pytest.mark.parametrize("k_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("hinted", [False, True], ids=["plain-topk", "temporal-topk"])
def test_free_running_tcgen05_shared_key(k_dtype, hinted):
    """One key shared by the heads: the tcgen05 kernel (FP8: integer q splits exactly into its
    high e4m3 term, the low term is zero)."""
    wl = _wl("tcint", n_req=3, n0=6000, kv_heads=1, k_dtype=k_dtype, top_k=256, shuffle=True)
    _free_running(wl, "tcgen05", 8, hinted)


def test_free_running_mtp_four_rows_with_commit():
    """Four verifier rows: per-row selections, their union, every row's top-K over the union
    and the deferred replay of the accepted rows, free-running for 8 steps."""
    wl = _wl("mtpint", n_req=3, n0=6000, kv_heads=1, k_dtype="bf16", top_k=256, rows=4, mean_accept=2.4)
    _free_running(wl, "tcgen05", 8)


# ------------------------------------------------------------------ FP8 query range

@pytest.mark.parametrize("small", [1e-2, 1e-3, 1e-5])
def test_fp8_query_wide_in_row_range(small):
    """Each (row, head) query vector holds one element of 8 and the others N(0, small):
    the low e4m3 term, and the subnormal floor below it, carry the small elements."""
    wl = syn.Workload("fp8q", n_req=3, n_layers=1, n0=4000, n_heads=64, head_dim=128, kv_heads=1,
                      q_dtype="bf16", k_dtype="e4m3", top_k=256, rho_bp=4000, gamma_bp=500, alpha=0.9,
                      steps=3, heavy=8, rope_dims=64, shuffle=True, seed=17)
    h = Harness(wl, score_path="tcgen05")
    g = torch.Generator(device="cuda").manual_seed(4)
    for step in range(3):
        _, w, qp = h.inp.step_inputs()
        q = torch.randn((3, 1, 64, 128), generator=g, device="cuda") * small
        col = torch.randint(0, 128, (3, 1, 64), generator=g, device="cuda")
        q.scatter_(3, col[..., None], 8.0)
        out = h.step(step, 0, q.to(torch.bfloat16), w, qp)
        h.inp.advance(step)
    assert out["worst"] < 2e-2
