"""Helpers of the GPU-vs-oracle parity tests.

Teacher-forced checking of one decode step of one layer: the oracle is fed the GPU's
pre-step state and must pick exactly the GPU's blocks; the GPU's scores must match the
oracle's within the stated tolerance (|dz| <= tol * sum_h |w_h| |s_i| sum_c |q k|); the
oracle's top-K of the GPU's scores must equal the GPU's top-K; the oracle's EMA update
from the GPU's pre-state and scores must equal the GPU's post-state bit for bit; and
Vmax must equal the blockwise max of V.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import oracle as o
from sparse_attention_indexer_spin_gb300 import spin
from sparse_attention_indexer_spin_gb300 import synthetic as syn

# Score tolerance: 1e-3 relative to the magnitude bound for fp32/bf16 inputs, 2e-2 for FP8
# keys (the stated bar; the kernels accumulate in fp32).
TOL = {"f32": 1e-3, "bf16": 1e-3, "e4m3": 2e-2}


def np_(t):
    return syn.raw_numpy(t)


class Harness:
    def __init__(self, wl: syn.Workload, score_path="auto", device="cuda", n0=None, layers=None):
        self.wl = wl
        self.inp = syn.SyntheticInputs(wl, device, layers=layers, n0=n0)
        self.cfg = spin.make_config(**wl.config_fields(), score_path=score_path)
        self.ocfg = o.make_cfg(**wl.config_fields())
        self.states = [spin.LayerState(self.cfg, device) for _ in range(self.inp.n_layers)]
        for s in self.states:
            spin.init_state(self.cfg, s.V, s.D, s.Vmax, s.warm)
        self.buf = spin.StepBuffers(self.cfg, wl.rows, device)
        self.tol = TOL[wl.k_dtype]
        # block-age exploration: the ages (uint32 bit patterns in an int32 tensor), one array per layer
        self.ages = None
        if wl.explore == "age":
            self.ages = [torch.zeros((wl.n_req, self.cfg.max_blocks), dtype=torch.int32, device=device)
                         for _ in range(self.inp.n_layers)]

    def step(self, step, layer, q, w, qp, rho_override=None, accepted=None, check=True,
             score_requests=None, hint=None):
        wl, cfg, st, buf, inp = self.wl, self.cfg, self.states[layer], self.buf, self.inp
        rows = wl.rows
        pre = dict(V=np_(st.V).copy(), D=np_(st.D).copy(), warm=np_(st.warm).copy())
        age = None if self.ages is None else self.ages[layer]
        pre_age = None if age is None else np_(age).view(np.uint32).copy()
        ns = np_(inp.n_slots).copy()
        qpn = np_(qp).copy()
        buf.status.zero_()
        spin.run_step(cfg, st, buf, q, w, inp.k_pool[layer], inp.k_scale[layer], inp.n_pages,
                      inp.block_table, inp.n_slots, qp, step, layer, rho_override, accepted,
                      hint=hint, block_age=age)
        torch.cuda.synchronize()
        if not check:
            return None
        rho = -1 if rho_override is None else int(rho_override.item())
        gb, gnb = np_(buf.blocks), np_(buf.n_blocks)
        ob, onb, ou, onu, ok = o.select_blocks(self.ocfg, pre["V"], pre["D"], pre["warm"], ns, qpn,
                                               rows, rho, step, layer, age=pre_age)
        assert ok
        np.testing.assert_array_equal(gnb, onb)
        for r in range(wl.n_req):
            for k in range(rows):
                np.testing.assert_array_equal(gb[r, k, : gnb[r, k]], ob[r, k, : onb[r, k]])
        if rows > 1:
            gu, gnu = np_(buf.union), np_(buf.n_union)
            np.testing.assert_array_equal(gnu, onu)
            for r in range(wl.n_req):
                np.testing.assert_array_equal(gu[r, : gnu[r]], ou[r, : onu[r]])
            blist, nlist = gu, gnu
        else:
            blist, nlist = np.ascontiguousarray(gb[:, 0, :]), np.ascontiguousarray(gnb[:, 0])
        gsc = np_(buf.scores)
        # scores: full check on the sampled requests (all by default)
        reqs = range(wl.n_req) if score_requests is None else score_requests
        worst = self.check_scores(layer, q, w, blist, nlist, ns, gsc, reqs)
        # top-K of the GPU's own scores
        oidx, ok = o.topk(self.ocfg, gsc, blist, nlist, ns, rows)
        assert ok
        np.testing.assert_array_equal(np_(buf.topk), oidx)
        # EMA from the GPU pre-state and scores
        if rows == 1 or accepted is not None:
            V1, D1, W1 = pre["V"].copy(), pre["D"].copy(), pre["warm"].copy()
            acc = None if accepted is None else np_(accepted)
            assert o.replay_ema(self.ocfg, V1, D1, W1, gsc, blist, nlist, ns, qpn, rows, acc)
            gV, gD = np_(st.V), np_(st.D)
            assert gV.tobytes() == V1.tobytes(), "V differs"
            assert gD.tobytes() == D1.tobytes(), "D differs"
            np.testing.assert_array_equal(np_(st.warm), W1)
            if wl.pooling != "a2":  # A2 keeps block-level state and no Vmax
                self.check_vmax(layer)
            if pre_age is not None:  # the listed blocks' ages: step + 1
                assert o.block_age_update(self.ocfg, pre_age, blist, nlist, ns, step)
                np.testing.assert_array_equal(np_(age).view(np.uint32), pre_age)
        assert int(buf.status.item()) == 0, "status %#x" % int(buf.status.item())
        return dict(blocks=gb, n_blocks=gnb, blist=blist, nlist=nlist, scores=gsc,
                    topk=np_(buf.topk), worst=worst)

    def check_vmax(self, layer):
        st = self.states[layer]
        V = np_(st.V)
        MB = self.cfg.max_blocks
        pad = np.zeros((V.shape[0], MB * 64), dtype=np.float32)
        pad[:, : V.shape[1]] = V
        want = pad.reshape(V.shape[0], MB, 64).max(-1)
        got = np_(st.Vmax)
        # Vmax is refreshed for every block that was ever updated; others stay 0 == max(0s)
        np.testing.assert_array_equal(got, want)

    def request_inputs(self, layer, r):
        """One request's whole context as a compact pool with an identity block table."""
        inp, MB = self.inp, self.cfg.max_blocks
        pages = inp.block_table[r].long()
        pool = np_(inp.k_pool[layer][pages])
        scale = None if inp.k_scale[layer] is None else np_(inp.k_scale[layer][pages])
        return pool, scale, np.arange(MB, dtype=np.int32)[None, :]

    def check_scores(self, layer, q, w, blist, nlist, ns, gsc, reqs):
        wl = self.wl
        ocfg1 = o.make_cfg(**{**wl.config_fields(), "n_req": 1})
        qn, wn = np_(q), np_(w)
        worst = 0.0
        for r in reqs:
            pool, scale, bt = self.request_inputs(layer, r)
            osc, mags, ok = o.indexer_score(ocfg1, qn[r:r + 1], wn[r:r + 1], pool, scale, bt,
                                            blist[r:r + 1], nlist[r:r + 1], ns[r:r + 1], wl.rows,
                                            want_mags=True)
            assert ok
            live = int(nlist[r]) * 64          # entries beyond the list hold stale values
            g = gsc[r:r + 1, :, :live].astype(np.float64)
            osc, mags = osc[:, :, :live], mags[:, :, :live]
            err = np.abs(g - osc.astype(np.float64))
            bound = self.tol * mags + 1e-30
            bad = err > bound
            assert not bad.any(), "score mismatch at %s: gpu %r oracle %r mag %r" % (
                np.argwhere(bad)[:3], g[bad][:3], osc[bad][:3], mags[bad][:3])
            if live:
                rel = err / np.maximum(mags, 1e-30)
                worst = max(worst, float(rel.max()))
        return worst
