"""Per-layer block budgets on top of the C ABI ("Sparse Attention Still Has a Dense Problem",
section "Per-layer block budgets", Figures 5-6).

Every `period` decoding steps a layer's step runs as a dense probe: a selection at the
budget floor gives the predicted block scores (the ranking every budget's selection uses),
then the step runs dense (sparsity 0, every block scored, the EMA updated from all of them)
and its top-K is the dense top-K.
spin_miss_curve turns the two into the layer's miss curve; after a probe step
spin_allocate_budgets recomputes the per-layer sparsities, which are published to a device
table (one int32 per layer) by a copy ordered on the stream between steps, so a kernel never
sees the table change under it and a captured graph keeps reading the same address.  The
other steps pass table[layer] to spin_select_blocks as rho_override.

Marshalling only: the curves and the allocation run in libspin.so's host functions, every
step of the indexer path in its kernels.
"""
from __future__ import annotations

import numpy as np
import torch

from . import spin


class BudgetController:
    def __init__(self, cfg, n_layers: int, target_rho_bp: int, period: int = 8, n_points: int = 101,
                 g_min: int = 0, device="cuda"):
        if n_points < 2 or 10000 % (n_points - 1):
            raise ValueError("n_points - 1 must divide 10000")
        unit = 10000 // (n_points - 1)
        if (10000 - target_rho_bp) % unit:
            raise ValueError("the target kept fraction must lie on the grid (%d bp steps)" % unit)
        self.cfg, self.n_layers, self.period, self.n_points = cfg, n_layers, period, n_points
        self.target_g = (10000 - target_rho_bp) // unit
        self.g_min = g_min
        self.table = torch.full((n_layers,), target_rho_bp, dtype=torch.int32, device=device)
        self._host = torch.empty((n_layers,), dtype=torch.int32).pin_memory()
        self._zero = torch.zeros((1,), dtype=torch.int32, device=device)
        self._sparse = torch.full((1,), 10000, dtype=torch.int32, device=device)
        self.curves = np.zeros((n_layers, n_points), np.float32)
        self.probed = np.zeros(n_layers, bool)
        self.g = np.full(n_layers, self.target_g, np.int32)
        self._copied = None  # event after the last table copy (its host buffer is reused)

    def is_probe(self, step: int) -> bool:
        return step % self.period == 0

    def rho_override(self, layer: int) -> torch.Tensor:
        return self.table[layer:layer + 1]

    def step(self, state, buf, q, w, k_pool, k_scale, n_pages, block_table, n_slots, q_pos, step, layer):
        """One layer's decode step (rows = 1): a dense probe on probe steps, else the budgeted
        step with the layer's entry of the device table."""
        if not self.is_probe(step):
            spin.run_step(self.cfg, state, buf, q, w, k_pool, k_scale, n_pages, block_table, n_slots, q_pos,
                          step, layer, self.rho_override(layer))
            return
        cfg = self.cfg
        R, MB = cfg.n_req, cfg.max_blocks
        warm = state.warm.cpu().numpy().copy()
        # predicted block scores: the selection writes them into the workspace unless its
        # budget covers every block, so it runs at sparsity 10000 (the budget floor); when
        # even that covers every block, every point of the curve keeps every block and the
        # scores do not matter.  Its selection is then overwritten by the dense step.
        spin.select_blocks(cfg, state.V, state.D, state.Vmax, state.warm, n_slots, q_pos, 1,
                           self._sparse, step, layer, buf.blocks, buf.n_blocks, None, None,
                           buf.workspace, buf.status)
        S = buf.workspace[: R * MB].view(R, MB).cpu().numpy().copy()
        spin.run_step(cfg, state, buf, q, w, k_pool, k_scale, n_pages, block_table, n_slots, q_pos, step, layer,
                      self._zero)
        topk = buf.topk[:, 0, :].cpu().numpy().copy()
        nb = (n_slots.cpu().numpy().astype(np.int64) + 63) // 64
        topk[warm == 0] = -1  # a cold request has no predictions to measure
        self.curves[layer] = spin.miss_curve(S, nb.astype(np.int32), topk, self.n_points)
        self.probed[layer] = True

    def publish(self):
        """Recompute the budgets from the layers' latest curves and copy them to the device
        table on the current stream (call between steps)."""
        if not self.probed.all():
            return
        self.g, rho = spin.allocate_budgets(self.curves, self.target_g, self.g_min)
        if self._copied is not None:
            self._copied.synchronize()
        self._host.copy_(torch.from_numpy(rho))
        self.table.copy_(self._host, non_blocking=True)
        self._copied = torch.cuda.Event()
        self._copied.record()
