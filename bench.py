#!/usr/bin/env python
"""Benchmark of the SPIN decode-time indexer step on GB300.

One step = one decode step of every layer of the workload: block selection, indexer score
over the selected blocks, top-K and EMA update (select -> score -> top-K -> commit for the
multi-row MTP workload), all through the C ABI.  Default workload: the DeepSeek-V3.2-like
indexer (1 request, 4 layers, 131072 slots, 64 heads x 128 dims, a bf16 key per head,
K = 2048) at 40 % target block sparsity.

Prints one JSON line.  `value` is scored slots per second over all ranks (scored slots =
slots of the selected blocks, times query rows); `e2e` repeats the measurement with the
step's inputs copied from pinned host memory and the top-K indices copied back inside the
timed region.  --impl reference times the CPU oracle instead (a bounded sample per step).

Multi-GPU: replicas only (the indexer step has no exchange between requests or layers);
each rank runs the whole workload on its own GPU.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from sparse_attention_indexer_spin_gb300 import synthetic as syn  # noqa: E402

FALLBACK_HBM_GBS = 6800.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=400)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["spin", "reference"], default="spin")
    p.add_argument("--config", default="v32", choices=sorted(syn.CONFIGS))
    p.add_argument("--rho", type=int, default=None, help="target sparsity in basis points")
    p.add_argument("--combine", choices=["max", "sum"], default=None,
                   help="predicted slot score: max(V, D) (Eq. 1) or V + D")
    p.add_argument("--topk", choices=["auto", "hinted", "plain"], default="auto",
                   help="temporal top-K seeded by the previous step's threshold, the plain one, or "
                        "auto: the temporal one for one query row, the plain one for several")
    p.add_argument("--schedule", choices=["stacked", "serial"], default="stacked",
                   help="one selection and one EMA launch per step for all layers, or layer by layer")
    p.add_argument("--no-configs", action="store_true", help="skip the per-workload measurements")
    p.add_argument("--configs", default="pr1,v32,v4flash,mtp,serving")
    p.add_argument("--config-steps", type=int, default=20, help="timed steps per workload measurement")
    p.add_argument("--cpu-steps", type=int, default=32, help="oracle steps of the CPU baseline (about 10 s)")
    p.add_argument("--no-dense", action="store_true")
    p.add_argument("--layers", type=int, default=None, help="fewer layers (small profiling case)")
    p.add_argument("--n0", type=int, default=None, help="fewer slots per request (small profiling case)")
    return p.parse_args()


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.path = None
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        except Exception:
            uuid = None
        self.uuid = uuid

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "100"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def tensor_peak(k_dtype):
    """Dense tensor peak (TFLOP/s) for a contraction in k_dtype: the measured sustained bf16
    figure, times 2 for e4m3 (the nominal FP8 : bf16 ratio); the fallback without the file."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    base, kind = 1700.0, "fallback"
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        if "bf16_tflops_sustained" in d:
            base, kind = float(d["bf16_tflops_sustained"]), "measured (bf16 sustained)"
    if k_dtype == "e4m3":
        return 2.0 * base, kind + " x 2 for e4m3"
    return base, kind


def kernel_source_hash(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "sparse_attention_indexer_spin_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload, kernel_file, alg_bytes):
    """DRAM bytes (read + write) per launch of the score kernel: the ratio of DRAM traffic to
    algorithmic bytes measured by ncu on a reduced case of the same workload, scaled to this
    launch's algorithmic bytes; None unless the capture was taken on the current source."""
    path = os.path.join(ROOT, "profiles", "score_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("source_hash") != kernel_source_hash([kernel_file, "spin_common.cuh"]):
        return None
    r = e.get("traffic_per_alg_byte")
    return None if r is None else float(r) * alg_bytes


# ----------------------------------------------------------------------- CUDA workload

class StackedState:
    """The SPIN state of L layers stacked along a new outermost dimension (one PyTorch
    allocation per array); layer(l) gives a layer's slices for the single-layer calls."""

    def __init__(self, cfg, L):
        R, MB = cfg.n_req, cfg.max_blocks
        self.V = torch.zeros((L, R, cfg.max_slots), dtype=torch.float32, device="cuda")
        self.D = torch.zeros((L, R, cfg.d_len), dtype=torch.float32, device="cuda")
        self.Vmax = torch.zeros((L, R, MB), dtype=torch.float32, device="cuda")
        self.warm = torch.zeros((L, R), dtype=torch.int32, device="cuda")

    def layer(self, l):
        from sparse_attention_indexer_spin_gb300 import spin
        st = spin.LayerState.__new__(spin.LayerState)
        st.V, st.D, st.Vmax, st.warm = self.V[l], self.D[l], self.Vmax[l], self.warm[l]
        return st


class Workload:
    """One workload's inputs, state and buffers on the GPU, stepped through the C ABI.

    schedule "stacked": per step one selection launch for all layers, then every layer's score
    and top-K, then one EMA update (or MTP commit) launch for all layers; "serial": every
    layer's select -> score -> top-K -> EMA in turn.  topk "hinted": the score kernel collects
    the temporal top-K's candidates; "plain": the top-K reads every score."""

    def __init__(self, wl: syn.Workload, n_steps: int, rho_bp: int, share: "Workload" = None,
                 topk: str = "hinted", schedule: str = "stacked"):
        from sparse_attention_indexer_spin_gb300 import spin
        self.spin = spin
        if topk == "auto":
            topk = "hinted" if wl.rows == 1 else "plain"
        self.topk_mode, self.schedule = topk, schedule
        self.wl = wl = wl.replace(steps=max(wl.steps, n_steps), rho_bp=rho_bp)
        self.cfg = spin.make_config(**wl.config_fields())
        self.rows = wl.rows
        self.n_steps = n_steps
        if share is not None:
            # same inputs, own configuration and state (the other sparsities of a sweep)
            for k in ("inp", "L", "q", "w", "n_slots", "q_pos", "accepted"):
                setattr(self, k, getattr(share, k))
            self._alloc()
            return
        self.inp = syn.SyntheticInputs(wl, "cuda")
        self.L = self.inp.n_layers
        # per-step inputs: a ring of query sets, N and q positions for every step
        ring = min(n_steps, 32)
        self.q, self.w = [], []
        for _ in range(ring):
            ql, wl_ = [], []
            for _layer in range(self.L):
                q, w, _ = self.inp.step_inputs()
                ql.append(q)
                wl_.append(w)
            self.q.append(ql)
            self.w.append(wl_)
        ns, acc = [], []
        for s in range(n_steps):
            ns.append(self.inp.n_slots.clone())
            a = self.inp.draw_accepted().cuda() if self.rows > 1 else None
            acc.append(a)
            self.inp.advance(s, a)
        self.n_slots = torch.stack(ns)                          # [steps][R]
        self.q_pos = (self.n_slots - 1).clamp_min(0).to(torch.int32).contiguous()
        self.accepted = acc
        self._alloc()

    def _alloc(self):
        spin, n_steps, wl, L, rows = self.spin, self.n_steps, self.wl, self.L, self.rows
        self.state = StackedState(self.cfg, L)
        self.states = [self.state.layer(l) for l in range(L)]
        self.hints = None
        if self.topk_mode == "hinted" and self._hint_ok():
            self.hints = [spin.TopkHint(self.cfg, rows) for _ in range(L)]
        self.buf = spin.StepBuffers(self.cfg, rows)
        R, MB = wl.n_req, self.cfg.max_blocks
        self.scores = torch.zeros((L, R, rows, MB * 64), dtype=torch.float32, device="cuda")
        self.topk = torch.full((L, R, rows, self.cfg.top_k), -1, dtype=torch.int32, device="cuda")
        ws = spin.workspace_size(self.cfg, rows)
        self.workspace = torch.zeros(((L * ws + 255) // 256) * 64, dtype=torch.float32, device="cuda")
        # per (step, layer) selections so the scored-slot count can be read back afterwards
        self.blocks = torch.full((n_steps, L, R, rows, MB), -1, dtype=torch.int32, device="cuda")
        self.n_blocks = torch.zeros((n_steps, L, R, rows), dtype=torch.int32, device="cuda")
        self.unions = torch.full((n_steps, L, R, MB), -1, dtype=torch.int32, device="cuda")
        self.n_unions = torch.zeros((n_steps, L, R), dtype=torch.int32, device="cuda")
        self.reset()

    def _hint_ok(self):
        try:
            self.spin.topk_hint_size(self.cfg, self.rows)
            return True
        except self.spin.SpinError:
            return False

    def reset(self):
        for st in self.states:
            self.spin.init_state(self.cfg, st.V, st.D, st.Vmax, st.warm)
        for h in self.hints or []:
            h.reset()

    def hint_stats(self):
        if not self.hints:
            return None
        tot = {}
        for h in self.hints:
            for k, v in h.stats().items():
                tot[k] = tot.get(k, 0) + v
        return tot

    def launches_per_step(self):
        if self.schedule == "stacked":
            return 3 + 2 * self.L      # block scores + selection, L x (score, top-K), EMA
        return self.L * 5              # L x (block scores, selection, score, top-K, EMA)

    def lists(self, s, layer):
        if self.rows == 1:
            return self.blocks[s, layer, :, 0], self.n_blocks[s, layer, :, 0]
        return self.unions[s, layer], self.n_unions[s, layer]

    def score_topk(self, s, layer, q, w, ev=None):
        spin, cfg, inp, rows = self.spin, self.cfg, self.inp, self.rows
        ns = self.n_slots[s]
        lst, nl = self.lists(s, layer)
        hint = self.hints[layer] if self.hints else None
        sc, tk = self.scores[layer], self.topk[layer]
        if ev is not None:
            ev[0].record()
        if hint is None:
            spin.indexer_score(cfg, q, w, inp.k_pool[layer], inp.k_scale[layer], inp.n_pages,
                               inp.block_table, lst, nl, ns, rows, sc, self.buf.status)
        else:
            spin.indexer_score_ex(cfg, q, w, inp.k_pool[layer], inp.k_scale[layer], inp.n_pages,
                                  inp.block_table, lst, nl, ns, rows, sc, self.buf.status, hint)
        if ev is not None:
            ev[1].record()
        if hint is None:
            spin.topk(cfg, sc, lst, nl, ns, rows, tk, self.buf.status)
        else:
            spin.topk_hinted(cfg, sc, w, lst, nl, ns, rows, tk, hint, self.buf.status)
        if ev is not None:
            ev[2].record()

    def step(self, s, ev_score=None, q_override=None, w_override=None, on_topk=None):
        spin, cfg, rows, L = self.spin, self.cfg, self.rows, self.L
        ns, qp = self.n_slots[s], self.q_pos[s]
        st, status = self.state, self.buf.status
        qs = q_override if q_override is not None else self.q[s % len(self.q)]
        ws = w_override if w_override is not None else self.w[s % len(self.w)]
        if self.schedule == "stacked":
            spin.select_blocks_layers(cfg, L, 0, st.V, st.D, st.Vmax, st.warm, ns, qp, rows, None, s,
                                      self.blocks[s], self.n_blocks[s],
                                      self.unions[s] if rows > 1 else None,
                                      self.n_unions[s] if rows > 1 else None, self.workspace, status)
            for layer in range(L):
                ev = None if ev_score is None else (ev_score[0][layer], ev_score[1][layer], ev_score[2][layer])
                self.score_topk(s, layer, qs[layer], ws[layer], ev)
                if on_topk is not None:
                    on_topk(layer)
            if rows == 1:
                spin.update_ema_layers(cfg, L, st.V, st.D, st.Vmax, st.warm, self.scores,
                                       self.blocks[s, :, :, 0], self.n_blocks[s, :, :, 0], ns, qp, status)
            else:
                spin.commit_mtp_layers(cfg, L, st.V, st.D, st.Vmax, st.warm, self.scores, rows,
                                       self.unions[s], self.n_unions[s], ns, qp, self.accepted[s], status)
            return
        for layer in range(L):
            lst_st = self.states[layer]
            un, nu = (self.unions[s, layer], self.n_unions[s, layer]) if rows > 1 else (None, None)
            spin.select_blocks(cfg, lst_st.V, lst_st.D, lst_st.Vmax, lst_st.warm, ns, qp, rows, None, s, layer,
                               self.blocks[s, layer], self.n_blocks[s, layer], un, nu, self.buf.workspace,
                               status)
            ev = None if ev_score is None else (ev_score[0][layer], ev_score[1][layer], ev_score[2][layer])
            self.score_topk(s, layer, qs[layer], ws[layer], ev)
            if on_topk is not None:
                on_topk(layer)
            lst, nl = self.lists(s, layer)
            if rows == 1:
                spin.update_ema(cfg, lst_st.V, lst_st.D, lst_st.Vmax, lst_st.warm, self.scores[layer], lst, nl,
                                ns, qp, status)
            else:
                spin.commit_mtp(cfg, lst_st.V, lst_st.D, lst_st.Vmax, lst_st.warm, self.scores[layer], rows, lst,
                                nl, ns, qp, self.accepted[s], status)

    def capture_graph(self):
        """One stacked step captured in a CUDA graph over static input buffers: the decode step
        is read from device memory by the selection (spin_select_blocks_layers with a device
        step), so a replay serves any step once its inputs are copied in."""
        spin, cfg, rows, L = self.spin, self.cfg, self.rows, self.L
        # every input of a step packed in one device buffer (256-byte aligned pieces), so that a
        # step's inputs arrive with one copy: N, q positions, the step, accepted counts, q and w
        def pieces(s):
            out = [self.n_slots[s], self.q_pos[s], torch.full((1,), s, dtype=torch.int64, device="cuda")]
            if rows > 1:
                out.append(self.accepted[s])
            for layer in range(L):
                out += [self.q[s % len(self.q)][layer], self.w[s % len(self.w)][layer]]
            return out
        offs, off = [], 0
        for t in pieces(0):
            offs.append(off)
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        self.g_in = torch.zeros(off, dtype=torch.uint8, device="cuda")

        def views(buf):
            return [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                    for o, t in zip(offs, pieces(0))]

        self.g_src = []
        for s_ in range(self.n_steps):
            src = torch.zeros(off, dtype=torch.uint8, device="cuda")
            for v, t in zip(views(src), pieces(s_)):
                v.copy_(t)
            self.g_src.append(src)
        vs = views(self.g_in)
        self.g_ns, self.g_qp, self.g_step = vs[0], vs[1], vs[2]
        self.g_acc = vs[3] if rows > 1 else None
        k = 4 if rows > 1 else 3
        self.g_q = [vs[k + 2 * layer] for layer in range(L)]
        self.g_w = [vs[k + 2 * layer + 1] for layer in range(L)]
        blocks, nbk, un, nun = self.blocks[0], self.n_blocks[0], self.unions[0], self.n_unions[0]
        st, status, inp = self.state, self.buf.status, self.inp

        def body():
            spin.select_blocks_layers(cfg, L, 0, st.V, st.D, st.Vmax, st.warm, self.g_ns, self.g_qp, rows, None,
                                      self.g_step, blocks, nbk, un if rows > 1 else None,
                                      nun if rows > 1 else None, self.workspace, status)
            for layer in range(L):
                lst, nl = (blocks[layer, :, 0], nbk[layer, :, 0]) if rows == 1 else (un[layer], nun[layer])
                hint = self.hints[layer] if self.hints else None
                sc, tk = self.scores[layer], self.topk[layer]
                q, w = self.g_q[layer], self.g_w[layer]
                if hint is None:
                    spin.indexer_score(cfg, q, w, inp.k_pool[layer], inp.k_scale[layer], inp.n_pages,
                                       inp.block_table, lst, nl, self.g_ns, rows, sc, status)
                    spin.topk(cfg, sc, lst, nl, self.g_ns, rows, tk, status)
                else:
                    spin.indexer_score_ex(cfg, q, w, inp.k_pool[layer], inp.k_scale[layer], inp.n_pages,
                                          inp.block_table, lst, nl, self.g_ns, rows, sc, status, hint)
                    spin.topk_hinted(cfg, sc, w, lst, nl, self.g_ns, rows, tk, hint, status)
            if rows == 1:
                spin.update_ema_layers(cfg, L, st.V, st.D, st.Vmax, st.warm, self.scores, blocks[:, :, 0],
                                       nbk[:, :, 0], self.g_ns, self.g_qp, status)
            else:
                spin.commit_mtp_layers(cfg, L, st.V, st.D, st.Vmax, st.warm, self.scores, rows, un, nun,
                                       self.g_ns, self.g_qp, self.g_acc, status)

        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, capture_error_mode="relaxed"):
            body()
        torch.cuda.synchronize()

    def replay_steps(self, steps):
        """Replays of the captured step, each after one copy of that step's packed inputs;
        returns the elapsed ms (CUDA events on the stream around all of them)."""
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for s in steps:
            self.g_in.copy_(self.g_src[s])      # the step's inputs, one copy
            self.graph.replay()
        t1.record()
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    def scored_slots(self, steps, unique=False):
        """Slots scored per (step, layer) launch, from the recorded lists: times the query
        rows (the metric's count), or each slot once (unique=True, the key bytes read)."""
        out = []
        ns_all = self.n_slots.cpu().numpy()
        lists = (self.blocks[:, :, :, 0] if self.rows == 1 else self.unions).cpu().numpy()
        counts = (self.n_blocks[:, :, :, 0] if self.rows == 1 else self.n_unions).cpu().numpy()
        for s in steps:
            for layer in range(self.L):
                tot = 0
                for r in range(self.wl.n_req):
                    blks = lists[s, layer, r, : counts[s, layer, r]].astype(np.int64)
                    tot += int(np.minimum(64, ns_all[s, r] - 64 * blks).clip(min=0).sum())
                out.append(tot if unique else tot * self.rows)
        return out

    def realized_sparsity(self, steps):
        """1 - (blocks scored) / (blocks of the contexts), over the steps, layers and requests."""
        ns = self.n_slots.cpu().numpy().astype(np.int64)
        counts = (self.n_blocks[:, :, :, 0] if self.rows == 1 else self.n_unions).cpu().numpy()
        sel = tot = 0
        for s in steps:
            nb = (ns[s] + 63) // 64
            sel += int(counts[s].sum())
            tot += int(nb.sum()) * self.L
        return 1.0 - sel / max(tot, 1)

    def key_bytes_per_slot(self):
        wl = self.wl
        elt = {"f32": 4, "bf16": 2, "e4m3": 1}[wl.k_dtype]
        return wl.kv_heads * wl.head_dim * elt + (4 if wl.k_dtype == "e4m3" else 0)

    def step_alg_bytes(self, steps):
        """Algorithmic HBM bytes of each step: the keys (+ FP8 scales) of every scored slot
        once, one fp32 score per slot and row written, the EMA update of the scored slots
        (a score read per row, V and D read and written), and block prediction (Vmax and the
        256-byte D window of every block under max, V and D of every slot under sum)."""
        ns = self.n_slots.cpu().numpy().astype(np.int64)
        uniq = np.array(self.scored_slots(steps, unique=True), np.float64).reshape(len(steps), self.L)
        pred = 260 if self.wl.combine == "max" else 512
        out = []
        for i, s in enumerate(steps):
            nb = float(((ns[s] + 63) // 64).sum()) * self.L * self.rows
            slots = uniq[i].sum()
            out.append(slots * (self.key_bytes_per_slot() + 4 * self.rows + 4 * self.rows + 16) + nb * pred)
        return out


def time_steps(wk, steps, with_score_events=False, topk_ms=None):
    """Run `steps` (list of step indices); returns (elapsed ms, per-score-launch ms list).
    With score events the score and top-K launches are bracketed by CUDA events on the
    stream (which also cuts the launch chaining at them): used for those kernels' own times
    only; the top-K times are appended to `topk_ms` when given."""
    ev_sets = []
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for s in steps:
        ev = None
        if with_score_events:
            ev = tuple([torch.cuda.Event(enable_timing=True) for _ in range(wk.L)] for _ in range(3))
            ev_sets.append(ev)
        wk.step(s, ev)
    t1.record()
    torch.cuda.synchronize()
    score_ms = [a.elapsed_time(b) for ev in ev_sets for a, b in zip(ev[0], ev[1])]
    if topk_ms is not None:
        topk_ms.extend(a.elapsed_time(b) for ev in ev_sets for a, b in zip(ev[1], ev[2]))
    return t0.elapsed_time(t1), score_ms


def time_pure_dense(wk, W, K):
    """The "pure dense" indexer: score and top-K over every block, with no prediction, no
    selection and no EMA update.  `wk` must be a workload at sparsity 0 whose steps 0..W+K-1
    have run, so its stored lists hold every block of each step's context.  Returns the mean
    ms per step over steps W..W+K-1 after a warm-up pass over 0..W-1."""
    def run(steps):
        for s in steps:
            qs, ws = wk.q[s % len(wk.q)], wk.w[s % len(wk.w)]
            for layer in range(wk.L):
                wk.score_topk(s, layer, qs[layer], ws[layer])

    for h in wk.hints or []:
        h.reset()
    run(range(W))
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    run(range(W, W + K))
    t1.record()
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / K


def pure_dense_entry(wk, W, K, sparse_ms):
    """time_pure_dense as a JSON entry beside the dense step.  It only re-runs the score and
    top-K launches of steps already run; a failure is recorded in the entry rather than ending
    the benchmark."""
    try:
        ms = time_pure_dense(wk, W, K)
        return {"ms_per_step": ms, "latency_ratio": sparse_ms / ms}
    except Exception as e:  # noqa: BLE001 -- the entry is a side measurement
        return {"error": repr(e)[:200]}


def time_e2e(wk, steps):
    """Same steps with per-step inputs staged from pinned host memory and the top-K read
    back to pinned host memory inside the timed region."""
    L = wk.L
    host_q = [[q.cpu().pin_memory() for q in ql] for ql in wk.q]
    host_w = [[w.cpu().pin_memory() for w in wl_] for wl_ in wk.w]
    host_ns = wk.n_slots.cpu().pin_memory()
    dev_q = [torch.empty_like(q) for q in wk.q[0]]
    dev_w = [torch.empty_like(w) for w in wk.w[0]]
    host_topk = torch.empty(tuple(wk.topk.shape), dtype=torch.int32).pin_memory()
    h2d = sum(q.numel() * q.element_size() for q in host_q[0]) + \
        sum(w.numel() * w.element_size() for w in host_w[0]) + host_ns[0].numel() * 4
    d2h = host_topk.numel() * 4

    def read_back(layer):
        host_topk[layer].copy_(wk.topk[layer], non_blocking=True)

    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for s in steps:
        i = s % len(host_q)
        for layer in range(L):
            dev_q[layer].copy_(host_q[i][layer], non_blocking=True)
            dev_w[layer].copy_(host_w[i][layer], non_blocking=True)
        wk.n_slots[s].copy_(host_ns[s], non_blocking=True)
        wk.step(s, None, dev_q, dev_w, read_back)
    t1.record()
    torch.cuda.synchronize()
    return t0.elapsed_time(t1), h2d, d2h


def miss_rate(wk, steps):
    """Share of each step's dense top-K (every block scored with the same queries) that lies
    in blocks the step did not score, over the layers, requests and rows (not timed).  Runs
    the steps (which must follow the ones already run) and scores densely before each."""
    spin, cfg, rows, inp = wk.spin, wk.cfg, wk.rows, wk.inp
    R, MB = wk.wl.n_req, cfg.max_blocks
    full = torch.arange(MB, dtype=torch.int32, device="cuda").repeat(R, 1).contiguous()
    sc = torch.zeros((R, rows, MB * 64), dtype=torch.float32, device="cuda")
    tk = torch.full((R, rows, cfg.top_k), -1, dtype=torch.int32, device="cuda")
    missed = total = 0
    for s in steps:
        ns = wk.n_slots[s]
        nfull = ((ns.long() + 63) // 64).to(torch.int32)
        dense = []
        for layer in range(wk.L):
            q, w = wk.q[s % len(wk.q)][layer], wk.w[s % len(wk.w)][layer]
            spin.indexer_score(cfg, q, w, inp.k_pool[layer], inp.k_scale[layer], inp.n_pages, inp.block_table,
                               full, nfull, ns, rows, sc, wk.buf.status)
            spin.topk(cfg, sc, full, nfull, ns, rows, tk, wk.buf.status)
            dense.append(tk.cpu().numpy().copy())
        wk.step(s)
        for layer in range(wk.L):
            lst, nl = wk.lists(s, layer)
            lst, nl = lst.cpu().numpy(), nl.cpu().numpy()
            for r in range(R):
                chosen = np.zeros(MB + 1, bool)
                chosen[lst[r, : nl[r]]] = True
                ids = dense[layer][r].ravel()
                ids = ids[ids >= 0]
                missed += int((~chosen[ids // 64]).sum())
                total += len(ids)
    return missed / max(total, 1)


def reduce_over_ranks(ms, slots, dist, device):
    """Whole-job figures of a replicas-only run: the slowest rank's time and the slots that
    all ranks scored.  `dist` is torch.distributed (or None for one process)."""
    if dist is None:
        return float(ms), int(slots)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    n = torch.tensor([int(slots)], dtype=torch.int64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), int(n.item())


# --------------------------------------------------------------------- CPU (oracle)

def oracle_sample(wl: syn.Workload, inp_host, state, n_steps, blocks_per_step, seed_step=0):
    """Time the CPU oracle on a bounded sample of the workload: per step, the selection of
    one layer for request 0 over its whole context, then score, top-K and EMA over the
    first `blocks_per_step` selected blocks.  Returns (slots/s, seconds, slots)."""
    from oracle import oracle as o
    ocfg = o.make_cfg(**{**wl.config_fields(), "n_req": 1})
    V, D, warm = state
    pool, scale, bt, q_list, w_list, ns, qp = inp_host
    MB = o.max_blocks(ocfg)
    slots = 0
    t0 = time.perf_counter()
    for s in range(n_steps):
        blocks, nb, union, nu, _ = o.select_blocks(ocfg, V, D, warm, ns, qp, wl.rows, -1, seed_step + s, 0)
        lst = union if wl.rows > 1 else np.ascontiguousarray(blocks[:, 0])
        cnt = (nu if wl.rows > 1 else nb[:, 0]).copy()
        cnt[0] = min(int(cnt[0]), blocks_per_step)
        q, w = q_list[s % len(q_list)], w_list[s % len(w_list)]
        sc, _ = o.indexer_score(ocfg, q, w, pool, scale, bt, lst, cnt, ns, wl.rows)
        o.topk(ocfg, sc, lst, cnt, ns, wl.rows)
        acc = np.zeros(1, np.int32) if wl.rows > 1 else None
        o.replay_ema(ocfg, V, D, warm, sc, lst, cnt, ns, qp, wl.rows, acc)
        blk = lst[0, : cnt[0]].astype(np.int64)
        slots += int(np.minimum(64, int(ns[0]) - 64 * blk).clip(min=0).sum()) * wl.rows
    dt = time.perf_counter() - t0
    return slots / dt, dt, slots


def host_inputs_for_oracle(wk_or_inp, wl, layer=0):
    inp = wk_or_inp
    pages = inp.block_table[0].long()
    pool = syn.raw_numpy(inp.k_pool[layer][pages])
    scale = None if inp.k_scale[layer] is None else syn.raw_numpy(inp.k_scale[layer][pages])
    bt = np.arange(pages.numel(), dtype=np.int32)[None, :]
    return pool, scale, bt


def workload_label(wl, n_layers, n0, rho):
    """The workload as both arms name it in their JSON line's config."""
    return ("%s: %d req x %d layers, %d slots, %d heads x %d, kv_heads %d, %s keys, K=%d, rho=%.0f%%, "
            "gamma=%.0f%%, rows=%d" % (wl.name, wl.n_req, n_layers, n0, wl.n_heads, wl.head_dim, wl.kv_heads,
                                       wl.k_dtype, wl.top_k, rho / 100, wl.gamma_bp / 100, wl.rows))


def run_reference(args):
    """The CPU oracle arm: each step a bounded sample of the workload on host cores."""
    wl = syn.CONFIGS[args.config]
    rho = wl.rho_bp if args.rho is None else args.rho
    wl = wl.replace(rho_bp=rho)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = syn.SyntheticInputs(wl.replace(n_req=1), dev, layers=1)
    pool, scale, bt = host_inputs_for_oracle(inp, wl)
    q_list, w_list = [], []
    for _ in range(4):
        q, w, _ = inp.step_inputs()
        q_list.append(syn.raw_numpy(q))
        w_list.append(syn.raw_numpy(w))
    from oracle import oracle as o
    ocfg = o.make_cfg(**{**wl.config_fields(), "n_req": 1})
    V, D, warm = o.new_state(ocfg)
    ns = syn.raw_numpy(inp.n_slots).copy()
    qp = (ns - 1).astype(np.int32)
    bps = 64
    # warm-up: one dense initialising step on a cheap sample, then the W warm-up steps
    oracle_sample(wl, (pool, scale, bt, q_list, w_list, ns, qp), (V, D, warm), 1 + args.warmup, bps)
    rate, secs, slots = oracle_sample(wl, (pool, scale, bt, q_list, w_list, ns, qp), (V, D, warm),
                                      args.steps, bps, 1 + args.warmup)
    line = {
        "impl": "reference", "metric": "scored slots/s (SPIN indexer step)", "value": rate,
        "unit": "slots/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_label(wl, args.layers or wl.n_layers, args.n0 or wl.n0, rho),
                   "combine": wl.combine,
                   "sample": "request 0, layer 0, %d selected blocks per step" % bps},
        "cpu_baseline": {"kind": "oracle", "value": rate, "unit": "slots/s", "cores": 1,
                         "sample": "per step: selection over the full context of request 0 (layer 0), "
                                   "then score/top-K/EMA over its first %d selected blocks" % bps},
        "e2e": {"value": rate, "unit": "slots/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ------------------------------------------------------------------------------- main

def host_cpu():
    """Host core count and CPU model (the oracle's baseline runs on one of these cores)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() in ("Model name", "Model"):
                model = line.split(":", 1)[1].strip()
                if line.startswith("Model name"):
                    break
    except Exception:
        pass
    return {"nproc": os.cpu_count(), "cpu_model": model}


def measure_workload(base, rho, W, K, topk, schedule, share=None, score_events=True):
    """W warm-up steps then K timed steps at sparsity rho (basis points).  Returns the
    workload and a record of the timed region."""
    wk = Workload(base, W + K, rho, share=share, topk=topk, schedule=schedule)
    wk.reset()
    time_steps(wk, range(W))
    ms, _ = time_steps(wk, range(W, W + K))
    rec = {"rho_bp": rho, "ms_per_step": ms / K, "step_us_per_layer": 1000.0 * ms / K / wk.L}
    slots = wk.scored_slots(range(W, W + K))
    rec["slots_per_s"] = sum(slots) / (ms / 1000.0)
    rec["realized_sparsity"] = wk.realized_sparsity(range(W, W + K))
    peak, _ = measured_peaks()
    step_bytes = float(np.mean(wk.step_alg_bytes(range(W, W + K))))
    rec["step_hbm_frac"] = step_bytes / (ms / K / 1000.0) / 1e9 / peak
    rec["step_alg_bytes"] = step_bytes
    if score_events:
        # the score kernel's own launches, timed separately (events cut the launch chaining)
        wk.reset()
        time_steps(wk, range(W))
        tk_ms = []
        _, score_ms = time_steps(wk, range(W, W + K), with_score_events=True, topk_ms=tk_ms)
        rec["topk_us"] = 1000.0 * float(np.mean(tk_ms))
        avg = float(np.mean(score_ms))
        unique = wk.scored_slots(range(W, W + K), unique=True)
        alg = float(np.mean(unique)) * (wk.key_bytes_per_slot() + 4 * wk.rows)
        rec["score_us"] = 1000.0 * avg
        rec["score_alg_bytes"] = alg
        rec["score_frac"] = alg / (avg / 1000.0) / 1e9 / peak
        if wk.wl.kv_heads == 1:
            # the shared-key score is a contraction on the tensor cores: its algorithmic FLOPs
            # (2 n_h d per slot and row) against the measured sustained bf16 peak, or twice it
            # for FP8 keys (the nominal e4m3 : bf16 ratio)
            flops = float(np.mean(unique)) * 2.0 * wk.wl.n_heads * wk.wl.head_dim * wk.rows
            tpeak, tkind = tensor_peak(wk.wl.k_dtype)
            rec["score_tensor"] = {"achieved_tflops": flops / (avg / 1000.0) / 1e12, "peak_tflops": tpeak,
                                   "frac": flops / (avg / 1000.0) / 1e12 / tpeak, "peak_kind": tkind}
    rec["topk_hint"] = wk.hint_stats()
    return wk, rec


def measure_budgets(name, W, K, period=8):
    """Per-layer block budgets ("Per-layer block budgets" of the project page): every
    `period` steps each layer runs a dense probe (selection at the budget floor, dense step,
    miss curve), the budgets are re-allocated and published to a device table, and the other
    steps select with their layer's entry.  Timed over K steps against the same layer-by-layer
    steps with the uniform budget; host work of the probe steps (curves, allocation, the
    synchronising copies) is inside the timed region."""
    from sparse_attention_indexer_spin_gb300 import spin
    from sparse_attention_indexer_spin_gb300.budgets import BudgetController
    base = syn.CONFIGS[name]
    out = {"period": period, "target_rho_bp": base.rho_bp}
    for mode in ("uniform", "per_layer"):
        wk = Workload(base, W + K, base.rho_bp, topk="plain", schedule="serial")
        ctl = BudgetController(wk.cfg, wk.L, base.rho_bp, period=period) if mode == "per_layer" else None

        def run(steps):
            for s in steps:
                for layer in range(wk.L):
                    st = wk.states[layer]
                    q, w = wk.q[s % len(wk.q)][layer], wk.w[s % len(wk.w)][layer]
                    ns, qp = wk.n_slots[s], wk.q_pos[s]
                    if ctl is None:
                        spin.run_step(wk.cfg, st, wk.buf, q, w, wk.inp.k_pool[layer], wk.inp.k_scale[layer],
                                      wk.inp.n_pages, wk.inp.block_table, ns, qp, s, layer)
                    else:
                        ctl.step(st, wk.buf, q, w, wk.inp.k_pool[layer], wk.inp.k_scale[layer], wk.inp.n_pages,
                                 wk.inp.block_table, ns, qp, s, layer)
                if ctl is not None and ctl.is_probe(s):
                    ctl.publish()

        wk.reset()
        run(range(W))
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        run(range(W, W + K))
        t1.record()
        torch.cuda.synchronize()
        out[mode + "_ms_per_step"] = t0.elapsed_time(t1) / K
        if ctl is not None:
            out["layer_rho_bp"] = [int(x) for x in ctl.table.cpu().tolist()]
        del wk
        torch.cuda.empty_cache()
    out["per_layer_vs_uniform"] = out["per_layer_ms_per_step"] / out["uniform_ms_per_step"]
    return out


def run_config(name, W, K, topk, schedule, extra=()):
    """Every measurement of one workload: its sparsity sweep (or its target and 0), the dense
    ratio, realized sparsity and miss rate at its target.  Returns a per_config entry."""
    base = syn.CONFIGS[name]
    points = sorted(set(base.sweep or ()) | {base.rho_bp, 0})
    out = {"workload": name, "layers": base.n_layers, "n_req": base.n_req, "rows": base.rows,
           "k_dtype": base.k_dtype, "kv_heads": base.kv_heads, "top_k": base.top_k,
           "target_rho_bp": base.rho_bp, "combine": base.combine, "schedule": schedule, "topk": topk}
    first, recs = None, {}
    for rho in [base.rho_bp] + [p for p in points if p != base.rho_bp]:
        wk, rec = measure_workload(base, rho, W, K, topk, schedule, share=first, score_events=(rho in (base.rho_bp, 0)))
        if first is None:
            first = wk
            # miss rate of the target sparsity against the dense top-K of the same queries
            wm = Workload(base, W + 4, rho, share=wk, topk=topk, schedule=schedule)
            wm.reset()
            time_steps(wm, range(W))
            rec["miss_rate"] = miss_rate(wm, range(W, W + 4))
            del wm
            # the same step captured once in a CUDA graph and replayed (inputs copied in per step)
            wk.reset()
            time_steps(wk, range(W))
            wk.capture_graph()
            wk.replay_steps(range(W, 2 * W))
            rec["graph_ms_per_step"] = wk.replay_steps(range(W, W + K)) / K
            rec["graph_status"] = int(wk.buf.status.item())
            del wk.graph
        if rho == 0:
            rec["pure_dense"] = pure_dense_entry(wk, W, K, recs.get(base.rho_bp, rec)["ms_per_step"])
        if wk is not first:
            del wk
        recs[rho] = rec
    tgt, dense = recs[base.rho_bp], recs[0]
    out["target"] = tgt
    out["dense"] = dense
    out["dense_ratio"] = tgt["ms_per_step"] / dense["ms_per_step"]
    out["sweep_us_per_step"] = {str(p): 1000.0 * recs[p]["ms_per_step"] for p in points}
    for label, kw in extra:
        b2 = base.replace(**kw)
        _, r1 = measure_workload(b2, base.rho_bp, W, K, topk, schedule, share=None, score_events=False)
        _, r0 = measure_workload(b2, 0, W, K, topk, schedule, share=None, score_events=False)
        out[label] = {"target_ms_per_step": r1["ms_per_step"], "dense_ms_per_step": r0["ms_per_step"],
                      "dense_ratio": r1["ms_per_step"] / r0["ms_per_step"], **kw}
    del first
    torch.cuda.empty_cache()
    return out


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from sparse_attention_indexer_spin_gb300 import spin
    spin.lib()

    base = syn.CONFIGS[args.config]
    if args.layers is not None:
        base = base.replace(n_layers=args.layers)
    if args.n0 is not None:
        base = base.replace(n0=args.n0)
    if args.combine is not None:
        base = base.replace(combine=args.combine)
    rho = base.rho_bp if args.rho is None else args.rho
    W, K = max(args.warmup, 3), args.steps
    wk = Workload(base, W + K, rho, topk=args.topk, schedule=args.schedule)
    wl = wk.wl

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # ---------------------------------------------------------------- device-resident
    wk.reset()
    clocks = ClockSampler()
    clocks.start()
    time_steps(wk, range(W))
    barrier()
    ms, _ = time_steps(wk, range(W, W + K))
    barrier()
    clk = clocks.stop()
    slots_per_launch = wk.scored_slots(range(W, W + K))
    slots_total = sum(slots_per_launch)
    ms_max, slots_all = reduce_over_ranks(ms, slots_total, dist, "cuda")
    value = slots_all / (ms_max / 1000.0)
    ms_per_step = ms_max / K
    hint_stats = wk.hint_stats()
    realized = wk.realized_sparsity(range(W, W + K))
    peak, peak_kind = measured_peaks()
    step_bytes = float(np.mean(wk.step_alg_bytes(range(W, W + K))))

    # dominant kernel: the indexer score, its launches bracketed by events on the stream
    wk.reset()
    time_steps(wk, range(W))
    tk_ms = []
    _, score_ms = time_steps(wk, range(W, W + K), with_score_events=True, topk_ms=tk_ms)
    avg_score_ms = float(np.mean(score_ms))
    avg_topk_us = 1000.0 * float(np.mean(tk_ms))
    kbytes = wk.key_bytes_per_slot()
    unique_per_launch = wk.scored_slots(range(W, W + K), unique=True)
    # keys (+ FP8 scale) of every scored slot once, plus one fp32 score per slot and row
    alg_bytes = float(np.mean(unique_per_launch)) * (kbytes + 4 * wk.rows)
    achieved = alg_bytes / (avg_score_ms / 1000.0) / 1e9
    kernel_file = "spin_score_stream.cu" if wl.kv_heads > 1 else "spin_score_tc.cu"
    traffic = ncu_traffic(wl.name, kernel_file, alg_bytes)

    # ---------------------------------------------------------------- dense comparison
    dense = None
    if not args.no_dense and rho != 0:
        wd = Workload(base, W + K, 0, share=wk, topk=args.topk, schedule=args.schedule)
        time_steps(wd, range(W))
        msd, _ = time_steps(wd, range(W, W + K))
        dense = {"rho": 0.0, "ms_per_step": msd / K, "latency_ratio": (ms / K) / (msd / K),
                 "topk_hint": wd.hint_stats()}
        dense["pure_dense"] = pure_dense_entry(wd, W, K, ms / K)
        del wd
        torch.cuda.empty_cache()

    # ---------------------------------------------------------------- end to end
    wk.reset()
    time_steps(wk, range(W))
    barrier()
    ms_e2e, h2d, d2h = time_e2e(wk, range(W, W + K))
    barrier()
    ms_e2e_max, _ = reduce_over_ranks(ms_e2e, slots_total, dist, "cuda")
    e2e_value = slots_all / (ms_e2e_max / 1000.0)

    # ---------------------------------------------------------------- CPU baseline
    cpu = None
    if rank == 0:
        pool, scale, bt = host_inputs_for_oracle(wk.inp, wl)
        q_list = [syn.raw_numpy(wk.q[i][0][:1]) for i in range(min(4, len(wk.q)))]
        w_list = [syn.raw_numpy(wk.w[i][0][:1]) for i in range(min(4, len(wk.w)))]
        st = wk.states[0]
        state = (syn.raw_numpy(st.V[:1]).copy(), syn.raw_numpy(st.D[:1]).copy(),
                 syn.raw_numpy(st.warm[:1]).copy())
        ns = syn.raw_numpy(wk.n_slots[W + K - 1][:1]).copy()
        qp = (ns - 1).astype(np.int32)
        bps = 256
        rate, secs, _ = oracle_sample(wl, (pool, scale, bt, q_list, w_list, ns, qp), state,
                                      args.cpu_steps, bps, W + K)
        cpu = {"kind": "oracle", "value": rate, "unit": "slots/s", "cores": 1, **host_cpu(),
               "sample": "%d steps of request 0, layer 0: selection over the full context, then "
                         "score/top-K/EMA over the first %d selected blocks (%.1f s)" % (args.cpu_steps, bps, secs)}
    status = int(wk.buf.status.item())
    launches = wk.launches_per_step() * K
    del wk
    torch.cuda.empty_cache()

    # ---------------------------------------------------------------- every workload
    per_config = None
    if not args.no_configs and rank == 0:
        per_config = {}
        Kc = max(3, min(K, args.config_steps))
        clocks2 = ClockSampler()
        clocks2.start()
        for name in args.configs.split(","):
            extra = (("sum_combiner", {"combine": "sum"}),) if name == "v32" else ()
            per_config[name] = run_config(name, W, Kc, args.topk, args.schedule, extra)
        if "v32" in per_config:
            # the one-layer-at-a-time schedule and the plain top-K, for comparison
            _, r_serial = measure_workload(syn.CONFIGS["v32"], 4000, W, Kc, args.topk, "serial", score_events=False)
            _, r_plain = measure_workload(syn.CONFIGS["v32"], 4000, W, Kc, "plain", args.schedule, score_events=False)
            per_config["v32"]["serial_schedule_ms_per_step"] = r_serial["ms_per_step"]
            per_config["v32"]["plain_topk_ms_per_step"] = r_plain["ms_per_step"]
            torch.cuda.empty_cache()
            # per-layer budgets with a dense probe every 8 steps (16 steps: two probes per layer)
            per_config["v32"]["budgets_probe_every_8"] = measure_budgets("v32", W, 16, period=8)
        per_config["clocks"] = clocks2.stop()

    if rank == 0:
        line = {
            "metric": "scored slots/s (SPIN indexer step)",
            "value": value,
            "unit": "slots/s",
            "n_gpus": world,
            "steps": K,
            "warmup": W,
            "ms_per_step": ms_per_step,
            "latency_us_per_layer_step": 1000.0 * ms_per_step / base.n_layers,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": wl.k_dtype if wl.k_dtype != "e4m3" else "e4m3/bf16",
            "data": "synthetic",
            "config": {"workload": workload_label(wl, base.n_layers, base.n0, rho),
                       "l2": "inputs larger than L2 (keys of every layer in their own pool, %.2f GB each)"
                             % (base.n_req * base.max_blocks * 64 * (wl.kv_heads * wl.head_dim *
                                {"f32": 4, "bf16": 2, "e4m3": 1}[wl.k_dtype]) / 1e9),
                       "combine": wl.combine, "schedule": args.schedule, "topk": args.topk,
                       "parallelism": "replicas" if world > 1 else "1 GPU"},
            "roofline": {"kernel": "indexer score (%s)" % kernel_file[:-3], "bound": "hbm",
                         "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_kind": peak_kind, "traffic": traffic,
                         "alg_bytes_per_launch": alg_bytes, "avg_launch_us": 1000.0 * avg_score_ms},
            "step_hbm": {"alg_bytes_per_step": step_bytes,
                         "frac": step_bytes / (ms_per_step / 1000.0) / 1e9 / peak, "peak": peak},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "slots/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches,
            "clocks": clk,
            "dense": dense,
            "realized_sparsity": realized,
            "topk": {"mode": args.topk, "hint": hint_stats, "avg_launch_us": avg_topk_us},
            "per_config": per_config,
            "status": status,
        }
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
