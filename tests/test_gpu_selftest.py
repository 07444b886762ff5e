"""The bounded wait of the pipelined kernels (spin_selftest_wait through the C ABI).

Every wait of a score kernel on its shared-memory stage barriers gives up after a limit of
GPU global time, or at once when another warp has raised the kernel's abort flag, and then
reports SPIN_STATUS_TIMEOUT instead of spinning on.  These tests run that wait on a barrier
nobody arrives on, with the abort flag raised, and with an arrival, and then check that the
next decode step on the same device is still correct (the context stayed usable).
"""
import pytest
import torch

from _parity import Harness
from sparse_attention_indexer_spin_gb300 import spin
from sparse_attention_indexer_spin_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

MS = 1000 * 1000


@pytest.fixture(scope="module", autouse=True)
def _lib(spin_lib):
    assert torch.cuda.is_available(), "these tests need a GPU"
    return spin_lib


def _run(mode, limit_ns):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(1, dtype=torch.int64, device="cuda")
    spin.selftest_wait(mode, limit_ns, status, elapsed)
    torch.cuda.synchronize()
    return int(status.item()), int(elapsed.item())


def test_wait_without_arrival_ends_at_its_limit():
    status, ns = _run(0, 50 * MS)
    assert status & spin.STATUS_BITS["TIMEOUT"]
    assert 50 * MS <= ns < 1000 * MS


def test_wait_with_abort_flag_ends_at_once():
    status, ns = _run(1, 5000 * MS)
    assert status & spin.STATUS_BITS["TIMEOUT"]
    assert ns < 50 * MS


def test_wait_with_arrival_succeeds():
    status, ns = _run(2, 1000 * MS)
    assert status == 0
    assert ns < 50 * MS


def test_context_usable_after_timeouts():
    _run(0, 20 * MS)
    _run(1, 20 * MS)
    h = Harness(syn.CONFIGS["pr1"].replace(steps=2, n_req=2))
    for step in range(2):
        q, w, qp = h.inp.step_inputs()
        h.step(step, 0, q, w, qp)
        h.inp.advance(step)


def test_selftest_rejects_bad_arguments():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(1, dtype=torch.int64, device="cuda")
    with pytest.raises(spin.SpinError):
        spin.selftest_wait(3, MS, status, elapsed)
    with pytest.raises(spin.SpinError):
        spin.selftest_wait(0, 0, status, elapsed)
