"""GPU parity of the stand-alone top-K call (through the C ABI) against the CPU oracle.

Each case picks the kernel the library dispatches to by its shape and drives a branch of it
with a score distribution: full radix passes, ties at the K-th score, a narrow range with
long shared leading bits, fewer live candidates than K, a sampled bracket with and without an
upper end, and a collection overflow that falls back to the full radix.  Indices are
compared bit-exactly (integer work: ties go to the lower slot id).
"""
import numpy as np
import pytest
import torch

from oracle import oracle as o
from sparse_attention_indexer_spin_gb300 import spin
from sparse_attention_indexer_spin_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(spin_lib):
    assert torch.cuda.is_available(), "these tests need a GPU"
    return spin_lib


def _fields(n_req, max_slots, rows, top_k):
    return dict(n_req=n_req, max_slots=max_slots, max_rows=rows, n_heads=8, head_dim=64, kv_heads=8,
                q_dtype="f32", k_dtype="f32", top_k=top_k, rho_bp=4000, gamma_bp=500, alpha=0.9)


# (n_req, max_slots, rows, top_k, dist, seed): the kernel each shape reaches is in the id
CASES = [
    pytest.param(3, 131072, 1, 2048, "normal", 1, id="cluster-normal"),
    pytest.param(3, 131072, 1, 2048, "ties", 2, id="cluster-ties"),
    pytest.param(2, 131072, 1, 2048, "narrow", 3, id="cluster-narrow"),
    pytest.param(4, 4000, 1, 2048, "normal", 4, id="cluster-fewer-than-K"),
    pytest.param(2, 65536, 4, 1024, "ties", 5, id="cluster-4rows"),
    pytest.param(32, 65536, 1, 2048, "normal", 6, id="sample-upper-end"),
    pytest.param(32, 131072, 1, 256, "normal", 7, id="sample-no-upper-end"),
    pytest.param(34, 131072, 1, 512, "ties", 8, id="sample-ties"),
    pytest.param(33, 131072, 1, 512, "narrow", 9, id="sample-narrow"),
    pytest.param(32, 65536, 1, 512, "equal", 10, id="sample-equal-overflow"),
    pytest.param(8, 65536, 4, 2048, "normal", 11, id="sample-4rows"),
    pytest.param(40, 12000, 1, 4096, "normal", 12, id="sample-small-lists"),
    pytest.param(32, 300000, 1, 512, "normal", 13, id="row-long-lists"),
    pytest.param(2, 400000, 1, 1024, "ties", 14, id="single-cta-long-lists"),
]


@pytest.mark.parametrize("n_req,max_slots,rows,top_k,dist,seed", CASES)
def test_topk_direct(n_req, max_slots, rows, top_k, dist, seed):
    f = _fields(n_req, max_slots, rows, top_k)
    cfg, ocfg = spin.make_config(**f), o.make_cfg(**f)
    scores, blist, n_list, n_slots = syn.topk_inputs(n_req, max_slots, rows, dist, seed)
    want, ok = o.topk(ocfg, scores, blist, n_list, n_slots, rows)
    assert ok
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = torch.full((n_req, rows, top_k), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    spin.topk(cfg, d(scores), d(blist), d(n_list), d(n_slots), rows, out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    np.testing.assert_array_equal(out.cpu().numpy(), want)


def test_topk_direct_repeatable():
    """The same call twice gives the same indices (no order depends on thread timing)."""
    f = _fields(3, 131072, 1, 2048)
    cfg = spin.make_config(**f)
    scores, blist, n_list, n_slots = syn.topk_inputs(3, 131072, 1, "ties", 21)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    s, b, nl, ns = d(scores), d(blist), d(n_list), d(n_slots)
    outs = []
    for _ in range(3):
        out = torch.full((3, 1, 2048), -7, dtype=torch.int32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        spin.topk(cfg, s, b, nl, ns, 1, out, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        outs.append(out.cpu().numpy())
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])
