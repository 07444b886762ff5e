"""The seeded synthetic input recipes (CPU): the stand-alone top-K inputs."""
import numpy as np
import pytest

from sparse_attention_indexer_spin_gb300 import synthetic as syn


@pytest.mark.parametrize("dist", ["normal", "ties", "narrow", "equal"])
def test_topk_inputs_recipe(dist):
    """The stand-alone top-K inputs: ascending lists holding the first and last block of each
    context, scores of the listed slots by the asked distribution, 1e30 past the context."""
    scores, blist, n_list, n_slots = syn.topk_inputs(5, 5000, 2, dist, 3)
    a, b, c, d = syn.topk_inputs(5, 5000, 2, dist, 3)
    assert np.array_equal(scores, a) and np.array_equal(blist, b)   # seeded
    assert np.array_equal(n_list, c) and np.array_equal(n_slots, d)
    for r in range(5):
        nb = (int(n_slots[r]) + 63) // 64
        lst = blist[r, : n_list[r]]
        assert lst[0] == 0 and lst[-1] == nb - 1 and np.all(np.diff(lst) > 0)
        assert np.all(blist[r, n_list[r]:] == -1)
        slot = (lst[:, None].astype(np.int64) * 64 + np.arange(64)[None, :]).ravel()
        z = scores[r, :, : n_list[r] * 64]
        assert np.all(z[:, slot >= n_slots[r]] == np.float32(1e30))
        live = z[:, slot < n_slots[r]]
        if dist == "equal":
            assert np.all(live == 0.5)
        elif dist == "ties":
            assert set(np.unique(live)) <= set(range(16))
        elif dist == "narrow":
            assert np.all((live >= 1.0) & (live < 1.0 + 2.0 ** -12 + 1e-7))
        assert np.all(scores[r, :, n_list[r] * 64:] == np.float32(1e30))
