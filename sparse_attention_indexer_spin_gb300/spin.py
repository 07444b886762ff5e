"""Thin ctypes binding of libspin.so (include/spin.h).

Argument marshalling only: every step of the SPIN indexer step runs in the library's CUDA
kernels.  Tensors are passed as raw device pointers on torch's current stream.  There is
no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB_PATH = os.path.join(PKG, "libspin.so")
HEADER = os.path.join(ROOT, "include", "spin.h")

DTYPE = {"f32": 0, "bf16": 1, "e4m3": 2}
COMBINE = {"max": 0, "sum": 1}
POOLING = {"max": 0, "mean": 1, "top4": 2, "slots": 3, "a2": 4}
EXPLORE = {"random": 0, "age": 1}
SCORE_PATH = {"auto": 0, "generic": 1, "stream": 2, "tcgen05": 3}

STATUS_BITS = {
    "BAD_N": 0x01, "BAD_QPOS": 0x02, "BAD_LIST": 0x04, "BAD_PAGE": 0x08,
    "BAD_ACCEPTED": 0x10, "TIMEOUT": 0x20, "BAD_RHO": 0x40,
}

ERRORS = {0: "SPIN_OK", 1: "SPIN_ERR_INVALID_ARG", 2: "SPIN_ERR_SHAPE", 3: "SPIN_ERR_CAPACITY",
          4: "SPIN_ERR_UNSUPPORTED", 5: "SPIN_ERR_CUDA"}


class SpinError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__("%s: %s" % (ERRORS.get(code, code), msg))
        self.code = code


class SpinScoreExtras(ctypes.Structure):
    _fields_ = [("topk_hint", ctypes.c_void_p), ("topk_hint_bytes", ctypes.c_size_t)]


class SpinConfig(ctypes.Structure):
    _fields_ = [
        ("n_req", ctypes.c_int32), ("max_slots", ctypes.c_int32), ("max_rows", ctypes.c_int32),
        ("block", ctypes.c_int32), ("n_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("kv_heads", ctypes.c_int32), ("q_dtype", ctypes.c_int32), ("k_dtype", ctypes.c_int32),
        ("top_k", ctypes.c_int32), ("rho_bp", ctypes.c_int32), ("gamma_bp", ctypes.c_int32),
        ("alpha", ctypes.c_float), ("combine", ctypes.c_int32), ("seed", ctypes.c_uint64),
        ("score_path", ctypes.c_int32), ("pooling", ctypes.c_int32), ("explore", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]

    @property
    def max_blocks(self) -> int:
        return (self.max_slots + self.block - 1) // self.block

    @property
    def d_len(self) -> int:
        return self.max_slots + self.max_rows


def make_config(n_req, max_slots, max_rows, n_heads, head_dim, kv_heads, q_dtype, k_dtype, top_k,
                rho_bp, gamma_bp, alpha, combine="max", seed=0, block=64, score_path="auto",
                pooling="max", explore="random", **_ignored) -> SpinConfig:
    return SpinConfig(int(n_req), int(max_slots), int(max_rows), int(block), int(n_heads),
                      int(head_dim), int(kv_heads), DTYPE[q_dtype], DTYPE[k_dtype], int(top_k),
                      int(rho_bp), int(gamma_bp), float(alpha), COMBINE[combine],
                      int(seed) & 0xFFFFFFFFFFFFFFFF, SCORE_PATH[score_path], POOLING[pooling],
                      EXPLORE[explore], 0)


def ensure_built() -> str:
    """Build the library in-tree if it is missing or stale (needs nvcc; no GPU needed)."""
    from . import build
    return build.build()


_LIB = None


def lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libspin.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64, u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
        C = ctypes.POINTER(SpinConfig)
        sig = {
            "spin_init_state": [C, P, P, P, P, i32, P],
            "spin_select_blocks": [C, P, P, P, P, P, P, i32, P, u64, i32, P, P, P, P, P,
                                   ctypes.c_size_t, P, P],
            "spin_select_blocks_noalloc": [C, P, P, P, P, P, P, i32, P, u64, i32, P, P, P, P, P, P],
            "spin_select_blocks_dstep": [C, P, P, P, P, P, P, i32, P, P, i32, P, P, P, P, P,
                                         ctypes.c_size_t, P, P],
            "spin_select_blocks_layers": [C, i32, i32, P, P, P, P, P, P, i32, P, u64, P, P, P, P, P,
                                          P, ctypes.c_size_t, P, P],
            "spin_update_ema_layers": [C, i32, P, P, P, P, P, P, P, P, P, P, P],
            "spin_commit_mtp_layers": [C, i32, P, P, P, P, P, i32, P, P, P, P, P, P, P],
            "spin_indexer_score": [C, P, P, P, P, i64, P, i64, P, P, P, i32, P, P, P],
            "spin_indexer_score_ex": [C, P, P, P, P, i64, P, i64, P, P, P, i32, P,
                                      ctypes.POINTER(SpinScoreExtras), P, P],
            "spin_topk_hint_size": [C, i32, ctypes.POINTER(ctypes.c_size_t)],
            "spin_init_topk_hint": [C, i32, P, ctypes.c_size_t, i32, P],
            "spin_topk_hinted": [C, P, P, P, P, P, i32, P, P, ctypes.c_size_t, P, P],
            "spin_topk": [C, P, P, P, P, i32, P, P, P],
            "spin_update_ema": [C, P, P, P, P, P, P, P, P, P, P, P],
            "spin_select_blocks_age": [C, P, P, P, P, P, P, i32, P, u64, i32, P, P, P, P, P, P,
                                       ctypes.c_size_t, P, P],
            "spin_update_ema_age": [C, P, P, P, P, P, P, P, P, P, P, u64, P, P],
            "spin_commit_mtp": [C, P, P, P, P, P, i32, P, P, P, P, P, P, P],
            "spin_workspace_size": [C, i32, ctypes.POINTER(ctypes.c_size_t)],
            "spin_selftest_wait": [i32, u64, P, P, P],
            "spin_miss_curve": [P, i32, i64, P, P, i32, i32, P],
            "spin_allocate_budgets": [P, i32, i32, i32, i32, P, P],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        L.spin_version.restype = ctypes.c_char_p
        L.spin_last_error_string.restype = ctypes.c_char_p
        _LIB = L
    return _LIB


def header_functions():
    """Names of the functions include/spin.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spin_[a-z_]+)\s*\(", text)))


def _check(rc: int):
    if rc != 0:
        raise SpinError(rc, lib().spin_last_error_string().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    assert t.is_cuda and t.is_contiguous(), "device tensors must be contiguous CUDA tensors"
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _host(a, dtype):
    """A C-contiguous numpy array of `dtype` (host functions take host arrays)."""
    import numpy as np
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, ctypes.c_void_p(a.ctypes.data)


def miss_curve(S, nb, topk, n_points=101):
    """One layer's miss curve over a batch (host arrays): S [n_req][stride] predicted block
    scores of a dense probe step, nb [n_req] blocks per context, topk [n_req][K] the probe's
    dense top-K.  Returns float32 [n_points]."""
    import numpy as np
    S, pS = _host(S, np.float32)
    nb, pnb = _host(nb, np.int32)
    topk, pk = _host(topk, np.int32)
    out = np.zeros(n_points, np.float32)
    _check(lib().spin_miss_curve(pS, S.shape[0], S.shape[1], pnb, pk, topk.shape[1], n_points,
                                 ctypes.c_void_p(out.ctypes.data)))
    return out


def allocate_budgets(miss, target_g, g_min=0):
    """Per-layer grid points and sparsities (basis points) from the layers' miss curves
    (host array [n_layers][n_points])."""
    import numpy as np
    miss, pm = _host(miss, np.float32)
    L, n_points = miss.shape
    g = np.zeros(L, np.int32)
    rho = np.zeros(L, np.int32)
    _check(lib().spin_allocate_budgets(pm, L, n_points, int(target_g), int(g_min),
                                       ctypes.c_void_p(g.ctypes.data), ctypes.c_void_p(rho.ctypes.data)))
    return g, rho


def selftest_wait(mode, limit_ns, status, elapsed_ns, stream=None):
    """spin_selftest_wait: the library's bounded barrier wait, with no arrival (mode 0), the
    abort flag raised (1) or an arrival (2)."""
    _check(lib().spin_selftest_wait(int(mode), int(limit_ns), _ptr(status), _ptr(elapsed_ns), _stream(stream)))


def version() -> str:
    return lib().spin_version().decode()


def workspace_size(cfg: SpinConfig, rows: int = 1) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().spin_workspace_size(ctypes.byref(cfg), rows, ctypes.byref(out)))
    return int(out.value)


def init_state(cfg, V, D, Vmax, warm, req=-1, stream=None):
    _check(lib().spin_init_state(ctypes.byref(cfg), _ptr(V), _ptr(D), _ptr(Vmax), _ptr(warm), req,
                                 _stream(stream)))


def select_blocks(cfg, V, D, Vmax, warm, n_slots, q_pos, rows, rho_override, step, layer, blocks,
                  n_blocks, union_blocks, n_union, workspace, status, stream=None):
    """`step` is an int, or a one-element int64 device tensor read by the kernels when they run
    (spin_select_blocks_dstep: a captured graph replays every step)."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if isinstance(step, torch.Tensor):
        assert step.dtype == torch.int64 and step.numel() == 1
        _check(lib().spin_select_blocks_dstep(
            ctypes.byref(cfg), _ptr(V), _ptr(D), _ptr(Vmax), _ptr(warm), _ptr(n_slots), _ptr(q_pos),
            rows, _ptr(rho_override), _ptr(step), int(layer), _ptr(blocks), _ptr(n_blocks),
            _ptr(union_blocks), _ptr(n_union), _ptr(workspace), ws_bytes, _ptr(status), _stream(stream)))
        return
    _check(lib().spin_select_blocks(
        ctypes.byref(cfg), _ptr(V), _ptr(D), _ptr(Vmax), _ptr(warm), _ptr(n_slots), _ptr(q_pos),
        rows, _ptr(rho_override), int(step), int(layer), _ptr(blocks), _ptr(n_blocks),
        _ptr(union_blocks), _ptr(n_union), _ptr(workspace), ws_bytes, _ptr(status), _stream(stream)))


def select_blocks_age(cfg, V, D, Vmax, warm, n_slots, q_pos, rows, rho_override, step, layer, block_age,
                      blocks, n_blocks, union_blocks, n_union, workspace, status, stream=None):
    """spin_select_blocks_age: block-age exploration; block_age is an int32 device tensor
    [R][MB] holding the uint32 ages."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().spin_select_blocks_age(
        ctypes.byref(cfg), _ptr(V), _ptr(D), _ptr(Vmax), _ptr(warm), _ptr(n_slots), _ptr(q_pos),
        rows, _ptr(rho_override), int(step), int(layer), _ptr(block_age), _ptr(blocks), _ptr(n_blocks),
        _ptr(union_blocks), _ptr(n_union), _ptr(workspace), ws_bytes, _ptr(status), _stream(stream)))


def update_ema_age(cfg, V, D, Vmax, warm, scores, list_, n_list, n_slots, q_pos, block_age, step, status,
                   stream=None):
    """spin_update_ema_age: the EMA update that also records the listed blocks' age."""
    _check(lib().spin_update_ema_age(ctypes.byref(cfg), _ptr(V), _ptr(D), _ptr(Vmax), _ptr(warm),
                                     _ptr(scores), _ptr(list_), _ptr(n_list), _ptr(n_slots), _ptr(q_pos),
                                     _ptr(block_age), int(step), _ptr(status), _stream(stream)))


def select_blocks_layers(cfg, n_layers, layer0, V, D, Vmax, warm, n_slots, q_pos, rows, rho_table,
                         step, blocks, n_blocks, union_blocks, n_union, workspace, status, stream=None):
    """Selections of n_layers stacked layers (arrays [L][...]) in one launch.  `step` is an int
    or a one-element int64 device tensor read when the kernels run."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    step_dev = step if isinstance(step, torch.Tensor) else None
    _check(lib().spin_select_blocks_layers(
        ctypes.byref(cfg), int(n_layers), int(layer0), _ptr(V), _ptr(D), _ptr(Vmax), _ptr(warm),
        _ptr(n_slots), _ptr(q_pos), rows, _ptr(rho_table), 0 if step_dev is not None else int(step),
        _ptr(step_dev), _ptr(blocks), _ptr(n_blocks), _ptr(union_blocks), _ptr(n_union),
        _ptr(workspace), ws_bytes, _ptr(status), _stream(stream)))


def update_ema_layers(cfg, n_layers, V, D, Vmax, warm, scores, list_, n_list, n_slots, q_pos, status,
                      stream=None):
    _check(lib().spin_update_ema_layers(ctypes.byref(cfg), int(n_layers), _ptr(V), _ptr(D), _ptr(Vmax),
                                        _ptr(warm), _ptr(scores), _ptr(list_), _ptr(n_list),
                                        _ptr(n_slots), _ptr(q_pos), _ptr(status), _stream(stream)))


def commit_mtp_layers(cfg, n_layers, V, D, Vmax, warm, scores, rows, union_blocks, n_union, n_slots,
                      q_pos, accepted, status, stream=None):
    _check(lib().spin_commit_mtp_layers(ctypes.byref(cfg), int(n_layers), _ptr(V), _ptr(D), _ptr(Vmax),
                                        _ptr(warm), _ptr(scores), rows, _ptr(union_blocks),
                                        _ptr(n_union), _ptr(n_slots), _ptr(q_pos), _ptr(accepted),
                                        _ptr(status), _stream(stream)))


def select_blocks_noalloc(cfg, V, D, Vmax, warm, n_slots, q_pos, rows, rho_override, step, layer,
                          blocks, n_blocks, union_blocks, n_union, status, stream=None):
    """spin_select_blocks without a workspace: for callers that cannot allocate device
    memory, the library's own static scratch array is used instead."""
    _check(lib().spin_select_blocks_noalloc(
        ctypes.byref(cfg), _ptr(V), _ptr(D), _ptr(Vmax), _ptr(warm), _ptr(n_slots), _ptr(q_pos),
        rows, _ptr(rho_override), int(step), int(layer), _ptr(blocks), _ptr(n_blocks),
        _ptr(union_blocks), _ptr(n_union), _ptr(status), _stream(stream)))


def indexer_score(cfg, q, w, k_pool, k_scale, n_pages, block_table, list_, n_list, n_slots, rows,
                  scores, status, stream=None):
    _check(lib().spin_indexer_score(
        ctypes.byref(cfg), _ptr(q), _ptr(w), _ptr(k_pool), _ptr(k_scale), int(n_pages),
        _ptr(block_table), block_table.shape[-1], _ptr(list_), _ptr(n_list), _ptr(n_slots), rows,
        _ptr(scores), _ptr(status), _stream(stream)))


def indexer_score_ex(cfg, q, w, k_pool, k_scale, n_pages, block_table, list_, n_list, n_slots, rows,
                     scores, status, topk_hint=None, stream=None):
    """spin_indexer_score_ex: the score kernel also collects the hinted top-K's candidates
    into `topk_hint` (a TopkHint)."""
    ex = SpinScoreExtras()
    if topk_hint is not None:
        ex.topk_hint = topk_hint.buf.data_ptr()
        ex.topk_hint_bytes = topk_hint.nbytes
    _check(lib().spin_indexer_score_ex(
        ctypes.byref(cfg), _ptr(q), _ptr(w), _ptr(k_pool), _ptr(k_scale), int(n_pages),
        _ptr(block_table), block_table.shape[-1], _ptr(list_), _ptr(n_list), _ptr(n_slots), rows,
        _ptr(scores), ctypes.byref(ex), _ptr(status), _stream(stream)))


def topk_hint_size(cfg: SpinConfig, rows: int = 1) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().spin_topk_hint_size(ctypes.byref(cfg), rows, ctypes.byref(out)))
    return int(out.value)


def init_topk_hint(cfg, rows, hint, req=-1, stream=None):
    _check(lib().spin_init_topk_hint(ctypes.byref(cfg), rows, _ptr(hint.buf), hint.nbytes, int(req),
                                     _stream(stream)))


def topk_hinted(cfg, scores, w, list_, n_list, n_slots, rows, topk_idx, hint, status, stream=None):
    _check(lib().spin_topk_hinted(ctypes.byref(cfg), _ptr(scores), _ptr(w), _ptr(list_), _ptr(n_list),
                                  _ptr(n_slots), rows, _ptr(topk_idx), _ptr(hint.buf), hint.nbytes,
                                  _ptr(status), _stream(stream)))


HINT_WORDS = 16
HINT_FIELDS = ("guess", "count", "extra", "hit", "miss", "overflow", "cold", "exact", "last")


class TopkHint:
    """Device buffer of the temporal top-K hint (allocated by PyTorch), zeroed on creation."""

    def __init__(self, cfg: SpinConfig, rows: int = 1, device="cuda"):
        self.cfg, self.rows = cfg, rows
        self.nbytes = topk_hint_size(cfg, rows)
        self.buf = torch.zeros(((self.nbytes + 255) // 256) * 256, dtype=torch.uint8, device=device)
        assert self.buf.data_ptr() % 256 == 0

    def reset(self, req=-1, stream=None):
        init_topk_hint(self.cfg, self.rows, self, req, stream)

    def records(self):
        """uint32 [n_req * rows][HINT_WORDS] copy of the records (synchronises)."""
        n = self.cfg.n_req * self.rows * HINT_WORDS
        return self.buf[: 4 * n].view(torch.int32).view(-1, HINT_WORDS).cpu().numpy().view("uint32")

    def stats(self):
        """Totals over all rows of the hit / miss / overflow / cold / exact counters."""
        r = self.records().astype("int64")
        return {f: int(r[:, i].sum()) for i, f in enumerate(HINT_FIELDS) if f in
                ("hit", "miss", "overflow", "cold", "exact")}


def topk(cfg, scores, list_, n_list, n_slots, rows, topk_idx, status, stream=None):
    _check(lib().spin_topk(ctypes.byref(cfg), _ptr(scores), _ptr(list_), _ptr(n_list),
                           _ptr(n_slots), rows, _ptr(topk_idx), _ptr(status), _stream(stream)))


def update_ema(cfg, V, D, Vmax, warm, scores, list_, n_list, n_slots, q_pos, status, stream=None):
    _check(lib().spin_update_ema(ctypes.byref(cfg), _ptr(V), _ptr(D), _ptr(Vmax), _ptr(warm),
                                 _ptr(scores), _ptr(list_), _ptr(n_list), _ptr(n_slots),
                                 _ptr(q_pos), _ptr(status), _stream(stream)))


def commit_mtp(cfg, V, D, Vmax, warm, scores, rows, union_blocks, n_union, n_slots, q_pos,
               accepted, status, stream=None):
    _check(lib().spin_commit_mtp(ctypes.byref(cfg), _ptr(V), _ptr(D), _ptr(Vmax), _ptr(warm),
                                 _ptr(scores), rows, _ptr(union_blocks), _ptr(n_union),
                                 _ptr(n_slots), _ptr(q_pos), _ptr(accepted), _ptr(status),
                                 _stream(stream)))


# ------------------------------------------------------------------------ convenience

class LayerState:
    """Device buffers of one layer's SPIN state (allocated by PyTorch)."""

    def __init__(self, cfg: SpinConfig, device="cuda"):
        R, MB = cfg.n_req, cfg.max_blocks
        self.V = torch.zeros((R, cfg.max_slots), dtype=torch.float32, device=device)
        self.D = torch.zeros((R, cfg.d_len), dtype=torch.float32, device=device)
        self.Vmax = torch.zeros((R, MB), dtype=torch.float32, device=device)
        self.warm = torch.zeros((R,), dtype=torch.int32, device=device)


class StepBuffers:
    """Per-step device buffers: selections, union, scores, top-K, workspace, status."""

    def __init__(self, cfg: SpinConfig, rows: int = 1, device="cuda"):
        R, MB = cfg.n_req, cfg.max_blocks
        self.rows = rows
        self.blocks = torch.full((R, rows, MB), -1, dtype=torch.int32, device=device)
        self.n_blocks = torch.zeros((R, rows), dtype=torch.int32, device=device)
        self.union = torch.full((R, MB), -1, dtype=torch.int32, device=device)
        self.n_union = torch.zeros((R,), dtype=torch.int32, device=device)
        self.scores = torch.zeros((R, rows, MB * 64), dtype=torch.float32, device=device)
        self.topk = torch.full((R, rows, cfg.top_k), -1, dtype=torch.int32, device=device)
        ws = workspace_size(cfg, rows)
        self.workspace = torch.zeros((ws + 255) // 256 * 64, dtype=torch.float32, device=device)
        self.status = torch.zeros((1,), dtype=torch.int32, device=device)

    @property
    def blist(self):
        return self.blocks[:, 0, :] if self.rows == 1 else self.union

    @property
    def n_list(self):
        return self.n_blocks[:, 0] if self.rows == 1 else self.n_union


def run_step(cfg, state: LayerState, buf: StepBuffers, q, w, k_pool, k_scale, n_pages,
             block_table, n_slots, q_pos, step=0, layer=0, rho_override=None, accepted=None,
             stream=None, hint: Optional[TopkHint] = None, block_age=None):
    """One decode step of one layer through the C ABI: select -> score -> top-K -> EMA
    (or, with rows > 1, select -> union -> score -> top-K -> deferred commit).  With a
    TopkHint the score kernel collects the temporal top-K's candidates and the hinted top-K
    replaces the plain one."""
    rows = buf.rows
    union = buf.union if rows > 1 else None
    n_union = buf.n_union if rows > 1 else None
    if block_age is None:
        select_blocks(cfg, state.V, state.D, state.Vmax, state.warm, n_slots, q_pos, rows,
                      rho_override, step, layer, buf.blocks, buf.n_blocks, union, n_union,
                      buf.workspace, buf.status, stream)
    else:
        select_blocks_age(cfg, state.V, state.D, state.Vmax, state.warm, n_slots, q_pos, rows,
                          rho_override, step, layer, block_age, buf.blocks, buf.n_blocks, union, n_union,
                          buf.workspace, buf.status, stream)
    if rows == 1:
        blist = buf.blocks            # row 0 list: stride MB per request
        nlist = buf.n_blocks
    else:
        blist, nlist = buf.union, buf.n_union
    if hint is None:
        indexer_score(cfg, q, w, k_pool, k_scale, n_pages, block_table, blist, nlist, n_slots, rows,
                      buf.scores, buf.status, stream)
        topk(cfg, buf.scores, blist, nlist, n_slots, rows, buf.topk, buf.status, stream)
    else:
        indexer_score_ex(cfg, q, w, k_pool, k_scale, n_pages, block_table, blist, nlist, n_slots,
                         rows, buf.scores, buf.status, hint, stream)
        topk_hinted(cfg, buf.scores, w, blist, nlist, n_slots, rows, buf.topk, hint, buf.status, stream)
    if rows == 1 and block_age is not None:
        update_ema_age(cfg, state.V, state.D, state.Vmax, state.warm, buf.scores, blist, nlist,
                       n_slots, q_pos, block_age, step, buf.status, stream)
    elif rows == 1:
        update_ema(cfg, state.V, state.D, state.Vmax, state.warm, buf.scores, blist, nlist,
                   n_slots, q_pos, buf.status, stream)
    elif accepted is not None:
        commit_mtp(cfg, state.V, state.D, state.Vmax, state.warm, buf.scores, rows, blist, nlist,
                   n_slots, q_pos, accepted, buf.status, stream)
