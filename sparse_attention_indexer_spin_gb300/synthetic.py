"""Seeded synthetic inputs shaped like the workloads of the SPIN paper.

This module generates inputs only; it holds none of the method's arithmetic (no EMA,
no block scoring, no selection, no indexer score).  Both the CUDA path's tests and
the oracle's tests draw their inputs from here.

Recipe (per request r, per layer l):
  * keys k_i ~ N(0, 1) over [kv_heads][d]; `heavy` slots drawn without replacement are
    scaled by 3 (the vertical lines of the paper's Figure 1);
  * RoPE (theta = 1e4, interleaved pairs) on the first `rope_dims` dims of every head at
    the slot's position i (the diagonal bands; the paper applies RoPE to half of each
    head's dims, §2);
  * FP8 keys: per-slot scale s_i = max|k_i| / 448 and codes e4m3(k_i / s_i);
  * queries: an AR(1) drift per request, q' = 0.95 q + sqrt(1 - 0.95^2) eps, with
    verifier row r one more AR(1) step after row r-1, then RoPE at position q_pos + r;
  * head weights w ~ U(0, 1), drawn fresh every step;
  * block table: request-contiguous pages, or one random permutation of all pages
    ("shuffled");
  * MTP acceptance: L = min(G, 4), G geometric on {1, 2, ...} with P(G > k) = c^k and
    1 + c + c^2 + c^3 = mean acceptance length; a = L - 1 accepted drafts.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

BLOCK = 64


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n_req: int
    n_layers: int
    n0: int               # slots per request at step 0
    n_heads: int
    head_dim: int
    kv_heads: int         # 1 = one key shared by all heads, n_heads = a key per head
    q_dtype: str          # "f32" | "bf16"
    k_dtype: str          # "f32" | "bf16" | "e4m3"
    top_k: int
    rho_bp: int           # target block sparsity (basis points)
    gamma_bp: int         # exploration share (basis points)
    alpha: float          # EMA decay
    steps: int
    rows: int = 1         # verifier query rows per step
    heavy: int = 16
    rope_dims: int = 32
    shuffle: bool = False
    grow_every: int = 1   # one new slot every `grow_every` steps (rows == 1)
    mean_accept: float = 0.0  # rows > 1: mean acceptance length
    combine: str = "max"
    pooling: str = "max"  # block reduction (max: Eq. 2; mean, top4, slots, a2: the ablations)
    explore: str = "random"  # exploration policy (random: the method; age: the block-age ablation)
    seed: int = 0
    sweep: tuple = ()

    @property
    def growth(self) -> int:
        if self.rows > 1:
            return self.steps * self.rows
        return (self.steps + self.grow_every - 1) // self.grow_every + 1

    @property
    def max_slots(self) -> int:
        return self.n0 + self.growth

    @property
    def max_blocks(self) -> int:
        return (self.max_slots + BLOCK - 1) // BLOCK

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def config_fields(self) -> dict:
        """Fields shared by the library's and the oracle's configuration structs."""
        return dict(n_req=self.n_req, max_slots=self.max_slots, max_rows=self.rows,
                    n_heads=self.n_heads, head_dim=self.head_dim, kv_heads=self.kv_heads,
                    q_dtype=self.q_dtype, k_dtype=self.k_dtype, top_k=self.top_k,
                    rho_bp=self.rho_bp, gamma_bp=self.gamma_bp, alpha=self.alpha,
                    combine=self.combine, pooling=self.pooling, explore=self.explore, seed=self.seed,
                    block=BLOCK)


# The five workloads.  Slot counts follow the paper's serving setup (507K cached + 5K
# new tokens compressed 4x -> 131072 slots), block size 64 and K in 512..2048.
CONFIGS = {
    "pr1": Workload("pr1", n_req=1, n_layers=1, n0=4096, n_heads=8, head_dim=64, kv_heads=8,
                    q_dtype="f32", k_dtype="f32", top_k=256, rho_bp=4000, gamma_bp=500,
                    alpha=0.9, steps=32, heavy=16, rope_dims=32, seed=0),
    "v32": Workload("v32", n_req=1, n_layers=4, n0=131072, n_heads=64, head_dim=128,
                    kv_heads=64, q_dtype="bf16", k_dtype="bf16", top_k=2048, rho_bp=4000,
                    gamma_bp=500, alpha=0.9, steps=64, heavy=256, rope_dims=64, seed=1,
                    sweep=(0, 2000, 4000)),
    "v4flash": Workload("v4flash", n_req=32, n_layers=1, n0=131072, n_heads=64, head_dim=128,
                        kv_heads=1, q_dtype="bf16", k_dtype="e4m3", top_k=512, rho_bp=4000,
                        gamma_bp=500, alpha=0.9, steps=128, heavy=256, rope_dims=64,
                        shuffle=True, grow_every=4, seed=2),
    "mtp": Workload("mtp", n_req=16, n_layers=1, n0=262144, n_heads=64, head_dim=128,
                    kv_heads=1, q_dtype="bf16", k_dtype="bf16", top_k=2048, rho_bp=4000,
                    gamma_bp=500, alpha=0.9, steps=256, rows=4, heavy=256, rope_dims=64,
                    mean_accept=2.4, seed=3),
    "serving": Workload("serving", n_req=96, n_layers=1, n0=131072, n_heads=64, head_dim=128,
                        kv_heads=1, q_dtype="bf16", k_dtype="e4m3", top_k=512, rho_bp=4000,
                        gamma_bp=500, alpha=0.9, steps=64, heavy=256, rope_dims=64,
                        shuffle=True, grow_every=4, seed=4, sweep=(0, 3000, 4000, 5000)),
}

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def _gen(device, *seed_parts) -> torch.Generator:
    s = 0x9E3779B1
    for p in seed_parts:
        s = (s * 1000003 + int(p) + 1) % (2 ** 61 - 1)
    g = torch.Generator(device=device)
    g.manual_seed(s)
    return g


def apply_rope(x: torch.Tensor, pos: torch.Tensor, rope_dims: int, theta: float = 1e4):
    """Rotate interleaved pairs (2p, 2p+1), p < rope_dims/2, of the last dim by pos*theta^(-2p/rope_dims).
    x: [..., n, d] float32, pos broadcastable to x.shape[:-1]."""
    if rope_dims <= 0:
        return x
    half = rope_dims // 2
    p = torch.arange(half, device=x.device, dtype=torch.float64)
    inv = theta ** (-2.0 * p / rope_dims)
    ang = pos.to(torch.float64).unsqueeze(-1) * inv          # [..., half]
    cos, sin = torch.cos(ang).to(x.dtype), torch.sin(ang).to(x.dtype)
    xr = x[..., :rope_dims].reshape(*x.shape[:-1], half, 2)
    a, b = xr[..., 0], xr[..., 1]
    out = x.clone()
    rot = torch.stack((a * cos - b * sin, a * sin + b * cos), dim=-1)
    out[..., :rope_dims] = rot.reshape(*x.shape[:-1], rope_dims)
    return out


def quantize_e4m3(k: torch.Tensor):
    """k: [slots, kv_heads, d] float32 -> (codes uint8 [slots, kv_heads, d], scale f32 [slots])."""
    amax = k.abs().amax(dim=(1, 2)).clamp_min(1e-30)
    scale = (amax / 448.0).to(torch.float32)
    codes = (k / scale[:, None, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return codes.view(torch.uint8), scale


def acceptance_ratio(mean_accept: float) -> float:
    """c in (0, 1) with 1 + c + c^2 + c^3 = mean_accept (bisection)."""
    lo, hi = 0.0, 1.0
    for _ in range(100):
        mid = 0.5 * (lo + hi)
        if 1 + mid + mid * mid + mid ** 3 < mean_accept:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


class SyntheticInputs:
    """All inputs of one workload on one device.

    Attributes: block_table int32 [R][MB]; k_pool[l] ([pages][64][kv_heads][d], dtype
    uint8 codes / bfloat16 / float32); k_scale[l] (float32 [pages][64] or None);
    n_slots int32 [R] (current N per request).
    """

    def __init__(self, wl: Workload, device="cpu", layers: Optional[int] = None,
                 n0: Optional[int] = None):
        self.wl = wl
        self.device = torch.device(device)
        self.n_layers = wl.n_layers if layers is None else layers
        R, MB = wl.n_req, wl.max_blocks
        self.n_pages = R * MB
        g = _gen("cpu", wl.seed, 1)
        if wl.shuffle:
            perm = torch.randperm(self.n_pages, generator=g).to(torch.int32)
        else:
            perm = torch.arange(self.n_pages, dtype=torch.int32)
        self.block_table = perm.reshape(R, MB).to(self.device)
        self.k_pool, self.k_scale = [], []
        for layer in range(self.n_layers):
            kp, ks = self._make_pool(layer)
            self.k_pool.append(kp)
            self.k_scale.append(ks)
        n_init = wl.n0 if n0 is None else n0
        self.n_slots = torch.full((R,), n_init, dtype=torch.int32, device=self.device)
        gq = _gen(self.device, wl.seed, 2)
        self.q_state = torch.randn((R, wl.n_heads, wl.head_dim), generator=gq,
                                   device=self.device, dtype=torch.float32)
        self._gq = gq
        self._ga = _gen("cpu", wl.seed, 3)
        self.accept_c = acceptance_ratio(wl.mean_accept) if wl.rows > 1 else 0.0

    # ------------------------------------------------------------------ keys
    def _make_pool(self, layer):
        wl, dev = self.wl, self.device
        R, MB, kvh, d = wl.n_req, wl.max_blocks, wl.kv_heads, wl.head_dim
        slots = MB * BLOCK
        if wl.k_dtype == "e4m3":
            pool = torch.empty((self.n_pages, BLOCK, kvh, d), dtype=torch.uint8, device=dev)
            scale = torch.empty((self.n_pages, BLOCK), dtype=torch.float32, device=dev)
        else:
            pool = torch.empty((self.n_pages, BLOCK, kvh, d), dtype=TORCH_DTYPE[wl.k_dtype],
                               device=dev)
            scale = None
        chunk = max(BLOCK, (1 << 24) // (kvh * d) // BLOCK * BLOCK)
        for r in range(R):
            g = _gen(dev, wl.seed, 100 + layer, r)
            gh = _gen("cpu", wl.seed, 200 + layer, r)
            heavy = torch.randperm(wl.n0, generator=gh)[: wl.heavy].to(dev)
            mult = torch.ones(slots, device=dev)
            mult[heavy] = 3.0
            pages = self.block_table[r].long()
            for s0 in range(0, slots, chunk):
                s1 = min(slots, s0 + chunk)
                k = torch.randn((s1 - s0, kvh, d), generator=g, device=dev, dtype=torch.float32)
                k = k * mult[s0:s1, None, None]
                pos = torch.arange(s0, s1, device=dev)[:, None].expand(s1 - s0, kvh)
                k = apply_rope(k, pos, wl.rope_dims)
                blk = torch.arange(s0, s1, device=dev) // BLOCK
                sl = torch.arange(s0, s1, device=dev) % BLOCK
                pg = pages[blk]
                if wl.k_dtype == "e4m3":
                    codes, sc = quantize_e4m3(k)
                    pool[pg, sl] = codes
                    scale[pg, sl] = sc
                else:
                    pool[pg, sl] = k.to(pool.dtype)
        return pool, scale

    # --------------------------------------------------------------- queries
    def step_inputs(self):
        """Queries and head weights of the current step (advances the query drift).
        Returns q [R][rows][n_h][d] (q_dtype), w float32 [R][rows][n_h], q_pos int32 [R]."""
        wl, dev = self.wl, self.device
        rho = 0.95
        c = math.sqrt(1.0 - rho * rho)
        eps = torch.randn(self.q_state.shape, generator=self._gq, device=dev)
        self.q_state = rho * self.q_state + c * eps
        rows = [self.q_state]
        for _ in range(1, wl.rows):
            e = torch.randn(self.q_state.shape, generator=self._gq, device=dev)
            rows.append(rho * rows[-1] + c * e)
        q = torch.stack(rows, dim=1)                                  # [R][rows][H][d]
        q_pos = (self.n_slots - 1).clamp_min(0)
        pos = (q_pos[:, None] + torch.arange(wl.rows, device=dev)[None, :])
        q = apply_rope(q, pos[:, :, None].expand(-1, -1, wl.n_heads), wl.rope_dims)
        q = q.to(TORCH_DTYPE[wl.q_dtype]).contiguous()
        w = torch.rand((wl.n_req, wl.rows, wl.n_heads), generator=self._gq, device=dev,
                       dtype=torch.float32)
        return q, w, q_pos.to(torch.int32).contiguous()

    def draw_accepted(self) -> torch.Tensor:
        """Accepted drafts a in [0, rows-1] per request (geometric acceptance length)."""
        wl = self.wl
        u = torch.rand(wl.n_req, generator=self._ga, dtype=torch.float64)
        # P(L >= k+1) = c^k  ->  L = 1 + floor(log(u)/log(c)), capped at rows
        if self.accept_c <= 0.0:
            L = torch.ones(wl.n_req, dtype=torch.int64)
        else:
            L = 1 + torch.floor(torch.log(u) / math.log(self.accept_c)).to(torch.int64)
        L = L.clamp(1, wl.rows)
        return (L - 1).to(torch.int32)

    def advance(self, step: int, accepted: Optional[torch.Tensor] = None):
        """Grow the context after a decode step."""
        wl = self.wl
        if wl.rows > 1:
            assert accepted is not None
            self.n_slots += accepted.to(self.device) + 1
        elif (step + 1) % wl.grow_every == 0:
            self.n_slots += 1
        self.n_slots.clamp_(max=wl.max_slots)


def raw_numpy(t: torch.Tensor):
    """Host numpy view of a tensor in the oracle's raw formats (bf16 -> uint16 bits)."""
    import numpy as np
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


TOPK_DISTS = ("normal", "ties", "narrow", "equal")


def topk_inputs(n_req: int, max_slots: int, rows: int, dist: str, seed: int, fill: float = 0.6):
    """Seeded inputs of a stand-alone top-K call (host numpy arrays):

    - n_slots: per request a context of max_slots/2 .. max_slots slots;
    - blist / n_list: an ascending list of a `fill` share of the context's blocks (the first
      and the last always listed);
    - scores [n_req][rows][MB*64]: the listed slots in list order, drawn from `dist`:
      'normal' (N(0, 1)), 'ties' (integers 0..15), 'narrow' (1 + 2^-12 * U[0, 1), many
      shared leading bits), 'equal' (all 0.5).  Slots at or beyond the context's end and
      entries past the list get 1e30, which no correct top-K may return.
    """
    import numpy as np
    rng = np.random.default_rng(seed)
    MB = (max_slots + 63) // 64
    n_slots = rng.integers(max_slots // 2, max_slots + 1, n_req).astype(np.int32)
    blist = np.full((n_req, MB), -1, np.int32)
    n_list = np.zeros(n_req, np.int32)
    scores = np.full((n_req, rows, MB * 64), 1e30, np.float32)
    for r in range(n_req):
        nb = (int(n_slots[r]) + 63) // 64
        k = max(1, min(nb, int(fill * nb)))
        pick = set(rng.choice(nb, k, replace=False).tolist()) | {0, nb - 1}
        lst = np.array(sorted(pick), np.int32)
        blist[r, : len(lst)] = lst
        n_list[r] = len(lst)
        C = len(lst) * 64
        slot = (lst[:, None].astype(np.int64) * 64 + np.arange(64)[None, :]).ravel()
        for row in range(rows):
            if dist == "normal":
                z = rng.standard_normal(C).astype(np.float32)
            elif dist == "ties":
                z = rng.integers(0, 16, C).astype(np.float32)
            elif dist == "narrow":
                z = (1.0 + rng.random(C) / 4096.0).astype(np.float32)
            elif dist == "equal":
                z = np.full(C, 0.5, np.float32)
            else:
                raise ValueError(dist)
            z[slot >= n_slots[r]] = 1e30
            scores[r, row, :C] = z
    return scores, blist, n_list, n_slots
