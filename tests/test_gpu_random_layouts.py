"""Seeded random layouts through the fused path, against the oracle.

Each case draws a handful of params -- tiny ones, ragged ones of a few
blocks, full-tile ones, narrow ones (C < 9, so rows are not 16-byte aligned)
and sometimes a 512-block full-tile param, which makes the layout cut launches
into full-tile and padding-aware runs -- a DP size and a rank.  The global
norm is summed over every rank's range (the pieces of each: whole params as
flat runs, whole row-block strips as spans, partial strips through the block
table), then the rank's fused step reads the row-major grads and writes the
row-major codes.  Everything is compared with the oracle: the norm within
1e-12, master / m / v / scales bit for bit, the codes byte for byte, and every
code outside the rank's range untouched.

"面向 Blockwise FP8 量化的 ZeRO 优化器设计" §块粒度切分 / §参数布局变换 / §总结;
"DeepSpeed ZeRO 优化" §七."""
import numpy as np
import pytest
import torch

import oracle
from blockwise_fp8_zero_fold_gb300 import fp8z1 as F
from tests._gpu import lib, to_host  # noqa: F401

pytestmark = pytest.mark.gpu
B = 16384
SENTINEL = 0x7F  # an E4M3 NaN code, which the step never writes


def _random_shapes(rng):
    shapes = []
    for _ in range(int(rng.integers(1, 7))):
        kind = int(rng.integers(0, 4))
        if kind == 0:
            r, c = rng.integers(1, 40, 2)
        elif kind == 1:
            r, c = rng.integers(100, 400, 2)
        elif kind == 2:
            r, c = 128 * rng.integers(1, 4, 2)
        else:
            r, c = rng.integers(1, 300), rng.integers(1, 9)
        shapes.append((int(rng.integers(1, 4)), int(r), int(c)))
    if rng.random() < 0.4:
        shapes.insert(int(rng.integers(0, len(shapes) + 1)), (1, 128 * 32, 128 * 16))  # 512 full tiles
    return shapes


@pytest.mark.parametrize("seed", range(12))
def test_random_layout_fused_step(lib, seed):
    rng = np.random.default_rng(1000 + seed)
    shapes = _random_shapes(rng)
    dp = int(rng.choice([1, 2, 3, 5]))
    rank = int(rng.integers(0, dp))
    L = F.fp8z1_build_layout(shapes, dp_size=dp)
    nblk = F.fp8z1_layout_info(L)[0]
    b0, b1 = F.fp8z1_shard_range(L, rank)
    assert (b0, b1) == oracle.shard_range(nblk, dp, rank)

    gh = [(rng.standard_normal(s) * 1024e-3).astype(np.float32) for s in shapes]
    ph = [(rng.standard_normal(s) * 0.02).astype(np.float32) for s in shapes]
    mh = [(rng.standard_normal(s) * 1e-4).astype(np.float32) for s in shapes]
    vh = [np.abs(rng.standard_normal(s) * 1e-8).astype(np.float32) for s in shapes]
    dg = [torch.from_numpy(x).cuda() for x in gh]
    gptrs = F.param_pointers(dg)

    # the global norm: every rank's partial, added as the all-reduce would
    s = torch.zeros(1, dtype=torch.float64, device="cuda")
    f = torch.zeros(1, dtype=torch.int32, device="cuda")
    for r in range(dp):
        a, b = F.fp8z1_shard_range(L, r)
        F.fp8z1_fold_norm(L, gptrs, None, a, b, s, f)
    og = oracle.fold(shapes, gh)
    os_, of = oracle.sumsq(og)
    torch.cuda.synchronize()
    assert f.item() == of == 0
    assert abs(s.item() - os_) <= 1e-12 * os_

    # the rank's state, folded by the oracle
    sl = slice(b0 * B, b1 * B)
    op, om, ov = (oracle.fold(shapes, x)[sl].copy() for x in (ph, mh, vh))
    dp_, dm, dv = (torch.from_numpy(x.copy()).cuda() for x in (op, om, ov))
    dsc = torch.full((b1 - b0,), -1.0, device="cuda")
    d8 = [torch.full(x.shape, SENTINEL, dtype=torch.uint8, device="cuda") for x in gh]
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=0.5, loss_scale=1024.0,
              step=int(rng.integers(1, 5)))
    F.fp8z1_step_fused(L, F.make_hp(**hp), d_grad_params=gptrs, master_shard=dp_, m_shard=dm, v_shard=dv,
                       d_fp8_params=F.param_pointers(d8), scale_shard=dsc, b0=b0, b1=b1, d_sumsq=s,
                       d_found_inf=f)
    torch.cuda.synchronize()
    q, osc, skipped = oracle.step(oracle.make_hp(**hp), os_, of, og[sl].copy(), op, om, ov)
    assert not skipped
    for got, want, what in [(dp_, op, "master"), (dm, om, "m"), (dv, ov, "v"), (dsc, osc, "scales")]:
        assert np.array_equal(to_host(got).view(np.uint32), want.view(np.uint32)), (what, shapes, dp, rank)
    want8 = [np.full(x.shape, SENTINEL, np.uint8) for x in gh]
    oracle.unfold(shapes, q, want8, b0, b1)
    for i, (got, want) in enumerate(zip(d8, want8)):
        assert np.array_equal(to_host(got), want), ("codes", i, shapes, dp, rank)
    assert F.fp8z1_device_status(L) == 0
