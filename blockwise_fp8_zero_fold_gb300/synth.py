"""Seeded synthetic inputs for the blockwise-FP8 ZeRO-1 step.

This module only draws random row-major tensors and describes the workloads;
it holds none of the method's arithmetic (no fold, norm, update or
quantisation).  Both the CUDA path and the CPU oracle take their inputs from
here, so the same seed gives both sides the same numbers.

Workloads (each tensor is a row-major float32 [E, R, C]; 2-D weights have E=1):

* ``tiny``   one 300x200 weight; DP=2, rank 0; 3 steps.
* ``dense``  qkv 4096x12288, o 4096x4096, gate_up 4096x28672, down 14336x4096
             and an unaligned 1000x3000; DP=1; grads with 0.1% outliers x100.
* ``moe``    32 experts of gate_up 7168x4096 and down 2048x7168 (3-D, the
             expert dim first); DP=8 rank 3, or the full buffer; 1% of the
             128x128 tiles all-zero in grad, master and both moments.
* ``ragged`` 4000 2-D tensors, R and C uniform in [17, 690] and never a
             multiple of 128; loss scale 65536, max_norm 0.8; +inf written
             into element (0, 0) of tensor 1234 on step 2.
* ``ragged_literal`` the same with R and C uniform in [17, 3000] (9.08 G
             real elements, 602268 blocks, about 160 GB on the device).
* ``large``  64 experts of 7168x4096 and 2048x7168 plus dense 7168x18432
             tensors (x9 for the 4.0 G-element reading, x4 for the literal list).

Stored grads are loss-scaled: grad = S * N(0, sigma) (exact, S a power of 2).
Distributions "N(0, s)" use s as the standard deviation; v = |N(0, s)|.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

TILE = 128  # side of the square weight tile the workloads zero out


@dataclasses.dataclass
class Workload:
    name: str
    shapes: List[Tuple[int, int, int]]
    dp: int = 1
    rank: int = 0
    steps: int = 3
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1
    max_norm: float = 1.0
    loss_scale: float = 1024.0
    growth_interval: int = 1000
    grad_sigma: float = 1e-3
    outlier_frac: float = 0.0
    outlier_mult: float = 100.0
    master_sigma: float = 0.02
    m_sigma: float = 0.0      # 0 -> zeros
    v_sigma: float = 0.0      # 0 -> zeros, else |N(0, v_sigma)|
    zero_tile_frac: float = 0.0
    inf_step: Optional[int] = None   # 1-based step whose grads get an +inf
    inf_param: int = 0
    seed: int = 0

    def hp(self):
        return dict(lr=self.lr, beta1=self.beta1, beta2=self.beta2, eps=self.eps,
                    weight_decay=self.weight_decay, max_norm=self.max_norm,
                    loss_scale=self.loss_scale)

    @property
    def n_real(self) -> int:
        return int(sum(e * r * c for e, r, c in self.shapes))


def ragged_shapes(n: int = 4000, lo: int = 17, hi: int = 690, seed: int = 0):
    """n 2-D shapes with R, C uniform in [lo, hi], redrawn while a multiple of 128."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        rc = []
        for _ in range(2):
            x = int(rng.integers(lo, hi + 1))
            while x % TILE == 0:
                x = int(rng.integers(lo, hi + 1))
            rc.append(x)
        out.append((1, rc[0], rc[1]))
    return out


def workload(name: str, **overrides) -> Workload:
    if name == "tiny":
        w = Workload("tiny", [(1, 300, 200)], dp=2, rank=0, steps=3, grad_sigma=1e-3)
    elif name == "dense":
        w = Workload("dense", [(1, 4096, 12288), (1, 4096, 4096), (1, 4096, 28672),
                               (1, 14336, 4096), (1, 1000, 3000)],
                     dp=1, rank=0, steps=10, grad_sigma=1e-4, outlier_frac=1e-3,
                     m_sigma=1e-4, v_sigma=1e-8)
    elif name == "moe":
        w = Workload("moe", [(32, 7168, 4096), (32, 2048, 7168)], dp=8, rank=3, steps=5,
                     grad_sigma=1e-4, m_sigma=1e-4, v_sigma=1e-8, zero_tile_frac=0.01)
    elif name in ("ragged", "ragged_literal"):
        hi = 690 if name == "ragged" else 3000
        w = Workload(name, ragged_shapes(hi=hi), dp=1, rank=0, steps=3, grad_sigma=1e-3,
                     loss_scale=65536.0, max_norm=0.8, inf_step=2, inf_param=1234)
    elif name in ("large", "large_literal"):
        dense = 9 if name == "large" else 4
        w = Workload(name, [(64, 7168, 4096), (64, 2048, 7168)] + [(1, 7168, 18432)] * dense,
                     dp=1, rank=0, steps=5, grad_sigma=5e-5, m_sigma=1e-4, v_sigma=1e-8)
    else:
        raise KeyError(name)
    return dataclasses.replace(w, **overrides)


# ---------------------------------------------------------------------------
# generators

_KIND_OFFSET = {"master": 1, "m": 2, "v": 3, "grad": 100, "tiles": 7, "outlier": 50}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _seed(w: Workload, kind: str, param: int, step: int = 0) -> int:
    return (w.seed * 1_000_003 + _KIND_OFFSET[kind] * 100_003 + step * 10_007 + param) & ((1 << 62) - 1)


def zero_tiles(w: Workload) -> List[torch.Tensor]:
    """Per param, the (e, tile_row, tile_col) triples of the 128x128 tiles that
    the workload sets to zero (int64 [k, 3]); empty when zero_tile_frac == 0."""
    out = []
    for i, (e, r, c) in enumerate(w.shapes):
        tr, tc = -(-r // TILE), -(-c // TILE)
        count = e * tr * tc
        k = int(round(w.zero_tile_frac * count))
        if k == 0:
            out.append(torch.zeros((0, 3), dtype=torch.int64))
            continue
        pick = torch.randperm(count, generator=_gen("cpu", _seed(w, "tiles", i)))[:k]
        pick, _ = torch.sort(pick)
        ee = pick // (tr * tc)
        rem = pick % (tr * tc)
        out.append(torch.stack([ee, rem // tc, rem % tc], dim=1))
    return out


def _apply_zero_tiles(t: torch.Tensor, tiles: torch.Tensor):
    for e, a, b in tiles.tolist():
        t[e, a * TILE:(a + 1) * TILE, b * TILE:(b + 1) * TILE] = 0


def _normal(shape, sigma, device, seed, out=None):
    t = out if out is not None else torch.empty(shape, dtype=torch.float32, device=device)
    assert tuple(t.shape) == tuple(shape) and t.dtype == torch.float32
    t.normal_(0.0, 1.0, generator=_gen(t.device, seed))
    if sigma != 1.0:
        t.mul_(sigma)
    return t


def make_state(w: Workload, kind: str, device="cpu") -> List[torch.Tensor]:
    """Row-major initial ``master``, ``m`` or ``v`` tensors of every param."""
    sigma = {"master": w.master_sigma, "m": w.m_sigma, "v": w.v_sigma}[kind]
    tiles = zero_tiles(w) if w.zero_tile_frac > 0 else None
    out = []
    for i, shp in enumerate(w.shapes):
        if sigma == 0.0:
            t = torch.zeros(shp, dtype=torch.float32, device=device)
        else:
            t = _normal(shp, sigma, device, _seed(w, kind, i))
            if kind == "v":
                t.abs_()
        if tiles is not None:
            _apply_zero_tiles(t, tiles[i])
        out.append(t)
    return out


def make_grads(w: Workload, step: int, device="cpu", out: Optional[Sequence[torch.Tensor]] = None):
    """Row-major loss-scaled grads of every param for 1-based ``step``.

    Fills ``out`` in place when given (to reuse device memory)."""
    tiles = zero_tiles(w) if w.zero_tile_frac > 0 else None
    res = []
    for i, shp in enumerate(w.shapes):
        o = out[i] if out is not None else None
        t = _normal(shp, w.grad_sigma, device, _seed(w, "grad", i, step), out=o)
        if w.outlier_frac > 0:
            mask = torch.rand(shp, generator=_gen(device, _seed(w, "outlier", i, step)),
                              device=device) < w.outlier_frac
            t[mask] *= w.outlier_mult
            del mask
        t.mul_(w.loss_scale)
        if tiles is not None:
            _apply_zero_tiles(t, tiles[i])
        if w.inf_step is not None and step == w.inf_step and i == w.inf_param:
            t[0, 0, 0] = float("inf")
        res.append(t)
    return res
