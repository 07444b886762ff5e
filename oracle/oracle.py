"""ctypes front end of the CPU oracle (oracle/spin_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, by __graft_entry__.smoke() and by the
CPU-baseline leg of bench.py, never by the library.  It imports numpy and ctypes only;
buffers cross as numpy arrays in the same layouts as the C ABI (see spin_oracle.h).

Element types of the raw inputs: float32 for "f32", uint16 bit patterns for "bf16",
uint8 codes for "e4m3"; the oracle decodes them itself.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

DTYPES = {"f32": 0, "bf16": 1, "e4m3": 2}
COMBINES = {"max": 0, "sum": 1}
POOLINGS = {"max": 0, "mean": 1, "top4": 2, "slots": 3, "a2": 4}
EXPLORES = {"random": 0, "age": 1}
RAW_NP = {"f32": np.float32, "bf16": np.uint16, "e4m3": np.uint8}


class OracleCfg(ctypes.Structure):
    _fields_ = [
        ("n_req", ctypes.c_int32),
        ("max_slots", ctypes.c_int32),
        ("max_rows", ctypes.c_int32),
        ("block", ctypes.c_int32),
        ("n_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("kv_heads", ctypes.c_int32),
        ("q_dtype", ctypes.c_int32),
        ("k_dtype", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("rho_bp", ctypes.c_int32),
        ("gamma_bp", ctypes.c_int32),
        ("alpha", ctypes.c_float),
        ("combine", ctypes.c_int32),
        ("seed", ctypes.c_uint64),
        ("pooling", ctypes.c_int32),
        ("explore", ctypes.c_int32),
    ]


_LIB = None


def lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, u64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
        C = ctypes.POINTER(OracleCfg)
        L.oracle_philox4x64_10.argtypes = [P, P, P]
        L.oracle_explore_key.argtypes = [u64, i32, u64, i32, i32, i64]
        L.oracle_explore_key.restype = ctypes.c_uint32
        L.oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
        L.oracle_decode_e4m3.restype = ctypes.c_double
        L.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
        L.oracle_decode_bf16.restype = ctypes.c_double
        L.oracle_budget.argtypes = [i64, i64, i64, i32]
        L.oracle_budget.restype = i64
        L.oracle_explore_count.argtypes = [i64, i64, i32]
        L.oracle_explore_count.restype = i64
        L.oracle_block_scores.argtypes = [C, P, P, i64, i64, P]
        L.oracle_select_blocks.argtypes = [C, P, P, P, P, P, i32, i32, u64, i32, P, P, P, P]
        L.oracle_select_blocks.restype = ctypes.c_int
        L.oracle_select_blocks_age.argtypes = [C, P, P, P, P, P, i32, i32, u64, i32, P, P, P, P, P]
        L.oracle_select_blocks_age.restype = ctypes.c_int
        L.oracle_block_age_update.argtypes = [C, P, P, P, P, u64]
        L.oracle_block_age_update.restype = ctypes.c_int
        L.oracle_indexer_score.argtypes = [C, P, P, P, P, i64, P, i64, P, P, P, i32, P, P]
        L.oracle_indexer_score.restype = ctypes.c_int
        L.oracle_score_slot.argtypes = [C, P, P, P, ctypes.c_float, i32, P, P]
        L.oracle_topk.argtypes = [C, P, P, P, P, i32, P]
        L.oracle_topk.restype = ctypes.c_int
        L.oracle_replay_ema.argtypes = [C, P, P, P, P, i32, P, P, P, P, P]
        L.oracle_replay_ema.restype = ctypes.c_int
        L.oracle_init_state.argtypes = [C, P, P, P, i32]
        _LIB = L
    return _LIB


def make_cfg(n_req, max_slots, max_rows, n_heads, head_dim, kv_heads, q_dtype, k_dtype,
             top_k, rho_bp, gamma_bp, alpha, combine="max", seed=0, block=64, pooling="max",
             explore="random", **_ignored):
    return OracleCfg(int(n_req), int(max_slots), int(max_rows), int(block), int(n_heads),
                     int(head_dim), int(kv_heads), DTYPES[q_dtype], DTYPES[k_dtype],
                     int(top_k), int(rho_bp), int(gamma_bp), float(alpha),
                     COMBINES[combine], int(seed) & 0xFFFFFFFFFFFFFFFF, POOLINGS[pooling],
                     EXPLORES[explore])


def max_blocks(cfg) -> int:
    return (cfg.max_slots + cfg.block - 1) // cfg.block


def d_len(cfg) -> int:
    return cfg.max_slots + cfg.max_rows


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "need a C-contiguous numpy array"
    return a.ctypes.data_as(ctypes.c_void_p)


def _arr(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


# ---------------------------------------------------------------- primitives

def philox4x64_10(ctr, key):
    c = np.array(ctr, dtype=np.uint64)
    k = np.array(key, dtype=np.uint64)
    out = np.zeros(4, dtype=np.uint64)
    lib().oracle_philox4x64_10(_p(c), _p(k), _p(out))
    return [int(x) for x in out]


def explore_key(seed, layer, step, row, req, j) -> int:
    return int(lib().oracle_explore_key(seed & 0xFFFFFFFFFFFFFFFF, layer, step, row, req, j))


def decode_e4m3(code: int) -> float:
    return float(lib().oracle_decode_e4m3(code))


def decode_bf16(bits: int) -> float:
    return float(lib().oracle_decode_bf16(bits))


def budget(n_blocks, top_k, rho_bp, block=64) -> int:
    return int(lib().oracle_budget(n_blocks, top_k, block, rho_bp))


def explore_count(m, n_forced, gamma_bp) -> int:
    return int(lib().oracle_explore_count(m, n_forced, gamma_bp))


def block_scores(cfg, V_req, D_req, n_slots, q):
    V_req = _arr(V_req, np.float32)
    D_req = _arr(D_req, np.float32)
    nb = (n_slots + cfg.block - 1) // cfg.block
    S = np.zeros(max(nb, 1), dtype=np.float32)
    lib().oracle_block_scores(ctypes.byref(cfg), _p(V_req), _p(D_req), n_slots, q, _p(S))
    return S[:nb]


# ---------------------------------------------------------------- the step

def select_blocks(cfg, V, D, warm, n_slots, q_pos, rows=1, rho_bp=-1, step=0, layer=0, age=None):
    """Returns (blocks [R][rows][MB], n_blocks [R][rows], union [R][MB], n_union [R], ok).
    age: the block ages [R][MB] (uint32) of block-age exploration."""
    R, MB = cfg.n_req, max_blocks(cfg)
    V = _arr(V, np.float32)
    D = _arr(D, np.float32)
    warm = _arr(warm, np.int32)
    n_slots = _arr(n_slots, np.int32)
    q_pos = _arr(q_pos, np.int32)
    blocks = np.full((R, rows, MB), -1, dtype=np.int32)
    n_blocks = np.zeros((R, rows), dtype=np.int32)
    union = np.full((R, MB), -1, dtype=np.int32)
    n_union = np.zeros(R, dtype=np.int32)
    if age is None:
        rc = lib().oracle_select_blocks(ctypes.byref(cfg), _p(V), _p(D), _p(warm), _p(n_slots),
                                        _p(q_pos), rows, rho_bp, step, layer, _p(blocks),
                                        _p(n_blocks), _p(union), _p(n_union))
    else:
        age = _arr(age, np.uint32)
        rc = lib().oracle_select_blocks_age(ctypes.byref(cfg), _p(V), _p(D), _p(warm), _p(n_slots),
                                            _p(q_pos), rows, rho_bp, step, layer, _p(age), _p(blocks),
                                            _p(n_blocks), _p(union), _p(n_union))
    return blocks, n_blocks, union, n_union, rc == 0


def block_age_update(cfg, age, blist, n_list, n_slots, step):
    """In place: age[req][blk] = step + 1 for every listed block (numpy uint32 [R][MB])."""
    assert age.dtype == np.uint32 and age.flags["C_CONTIGUOUS"]
    rc = lib().oracle_block_age_update(ctypes.byref(cfg), _p(age), _p(_arr(blist, np.int32)),
                                       _p(_arr(n_list, np.int32)), _p(_arr(n_slots, np.int32)), int(step))
    return rc == 0


def indexer_score(cfg, q, w, k_pool, k_scale, block_table, blist, n_list, n_slots, rows=1,
                  want_mags=False):
    """Scores [R][rows][MB*64] (and magnitudes) of every listed block."""
    R, MB = cfg.n_req, max_blocks(cfg)
    q = np.ascontiguousarray(q)
    w = _arr(w, np.float32)
    k_pool = np.ascontiguousarray(k_pool)
    k_scale = None if k_scale is None else _arr(k_scale, np.float32)
    block_table = _arr(block_table, np.int32)
    blist = _arr(blist, np.int32)
    n_list = _arr(n_list, np.int32)
    n_slots = _arr(n_slots, np.int32)
    slot_elems = cfg.kv_heads * cfg.head_dim
    n_pages = k_pool.size // (slot_elems * cfg.block)
    scores = np.zeros((R, rows, MB * cfg.block), dtype=np.float32)
    mags = np.zeros((R, rows, MB * cfg.block), dtype=np.float64) if want_mags else None
    rc = lib().oracle_indexer_score(ctypes.byref(cfg), _p(q), _p(w), _p(k_pool), _p(k_scale),
                                    n_pages, _p(block_table), block_table.shape[-1],
                                    _p(blist), _p(n_list), _p(n_slots), rows, _p(scores),
                                    _p(mags))
    if want_mags:
        return scores, mags, rc == 0
    return scores, rc == 0


def score_slot(cfg, q_req, w_req, key, scale=1.0, rows=1):
    q_req = np.ascontiguousarray(q_req)
    w_req = _arr(w_req, np.float32)
    key = np.ascontiguousarray(key)
    z = np.zeros(rows, dtype=np.float32)
    mag = np.zeros(rows, dtype=np.float64)
    lib().oracle_score_slot(ctypes.byref(cfg), _p(q_req), _p(w_req), _p(key), float(scale),
                            rows, _p(z), _p(mag))
    return z, mag


def topk(cfg, scores, blist, n_list, n_slots, rows=1):
    R = cfg.n_req
    scores = _arr(scores, np.float32)
    blist = _arr(blist, np.int32)
    n_list = _arr(n_list, np.int32)
    n_slots = _arr(n_slots, np.int32)
    out = np.full((R, rows, cfg.top_k), -1, dtype=np.int32)
    rc = lib().oracle_topk(ctypes.byref(cfg), _p(scores), _p(blist), _p(n_list), _p(n_slots),
                           rows, _p(out))
    return out, rc == 0


def replay_ema(cfg, V, D, warm, scores, blist, n_list, n_slots, q_pos, rows=1, accepted=None):
    """In-place EMA update of V, D, warm (numpy float32/int32 arrays)."""
    for a, dt in ((V, np.float32), (D, np.float32), (warm, np.int32)):
        assert a.dtype == dt and a.flags["C_CONTIGUOUS"]
    scores = _arr(scores, np.float32)
    blist = _arr(blist, np.int32)
    n_list = _arr(n_list, np.int32)
    n_slots = _arr(n_slots, np.int32)
    q_pos = _arr(q_pos, np.int32)
    acc = None if accepted is None else _arr(accepted, np.int32)
    rc = lib().oracle_replay_ema(ctypes.byref(cfg), _p(V), _p(D), _p(warm), _p(scores), rows,
                                 _p(blist), _p(n_list), _p(n_slots), _p(q_pos), _p(acc))
    return rc == 0


def init_state(cfg, V, D, warm, req=-1):
    lib().oracle_init_state(ctypes.byref(cfg), _p(V), _p(D), _p(warm), req)


def new_state(cfg):
    V = np.zeros((cfg.n_req, cfg.max_slots), dtype=np.float32)
    D = np.zeros((cfg.n_req, d_len(cfg)), dtype=np.float32)
    warm = np.zeros(cfg.n_req, dtype=np.int32)
    return V, D, warm


class OracleStep:
    """One full single-row or multi-row decode step of one layer, in the paper's order."""

    def __init__(self, cfg):
        self.cfg = cfg

    def run(self, V, D, warm, q, w, k_pool, k_scale, block_table, n_slots, q_pos, rows=1,
            step=0, layer=0, rho_bp=-1, accepted=None):
        cfg = self.cfg
        blocks, n_blocks, union, n_union, ok1 = select_blocks(
            cfg, V, D, warm, n_slots, q_pos, rows, rho_bp, step, layer)
        if rows == 1:
            blist, n_list = blocks[:, 0, :], n_blocks[:, 0]
        else:
            blist, n_list = union, n_union
        scores, ok2 = indexer_score(cfg, q, w, k_pool, k_scale, block_table, blist, n_list,
                                    n_slots, rows)
        idx, ok3 = topk(cfg, scores, blist, n_list, n_slots, rows)
        ok4 = replay_ema(cfg, V, D, warm, scores, blist, n_list, n_slots, q_pos, rows, accepted)
        return dict(blocks=blocks, n_blocks=n_blocks, union=union, n_union=n_union,
                    blist=np.ascontiguousarray(blist), n_list=np.ascontiguousarray(n_list),
                    scores=scores, topk=idx, ok=ok1 and ok2 and ok3 and ok4)
