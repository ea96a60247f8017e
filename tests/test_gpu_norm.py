"""GPU parity: global grad norm + inf/nan flag against the oracle's exact sum.

"DeepSpeed ZeRO 优化" §七 (sum of squares over all ranks, combined by an
all-reduce -- here the per-range partials of one buffer) and §六 / §九 Q6."""
import numpy as np
import pytest
import torch

import oracle
from blockwise_fp8_zero_fold_gb300 import fp8z1 as F
from tests._gpu import lib, to_host  # noqa: F401

pytestmark = pytest.mark.gpu

NBLK = 37  # several CTAs' worth plus an uneven split


def _norm(L, g, b0, b1, sumsq=None, found=None):
    sumsq = torch.zeros(1, dtype=torch.float64, device="cuda") if sumsq is None else sumsq
    found = torch.zeros(1, dtype=torch.int32, device="cuda") if found is None else found
    F.fp8z1_grad_norm(L, g[b0 * 16384:] if b0 else g, b0, b1, sumsq, found)
    torch.cuda.synchronize()
    return float(sumsq.item()), int(found.item()), sumsq, found


@pytest.fixture(scope="module")
def layout(lib):
    return F.fp8z1_build_layout([(NBLK, 128, 128)], dp_size=4)


@pytest.mark.parametrize("dist", ["normal", "scaled", "outliers", "wide", "tiny", "huge", "zeros"])
def test_sumsq_matches_exact(layout, dist):
    rng = np.random.default_rng(hash(dist) % 2**32)
    n = NBLK * 16384
    g = rng.standard_normal(n)
    if dist == "scaled":
        g *= 1e-4 * 1024
    elif dist == "outliers":
        g *= 1e-4
        g[rng.random(n) < 1e-3] *= 100
    elif dist == "wide":
        g *= np.exp2(rng.integers(-80, 70, n))
    elif dist == "tiny":
        g *= 1e-35           # squares underflow float32: the double path
    elif dist == "huge":
        g *= 1e25            # squares overflow float32: the double path
    elif dist == "zeros":
        g[:] = 0
    g = g.astype(np.float32)
    dg = torch.from_numpy(g).cuda()
    for b0, b1 in [(0, NBLK), (3, 20), (36, 37), (0, 1)]:
        got, found, _, _ = _norm(layout, dg, b0, b1)
        want, wf = oracle.sumsq(g[b0 * 16384:b1 * 16384])
        assert found == wf == 0
        if want == 0:
            assert got == 0
        else:
            assert abs(got - want) <= 1e-5 * want           # contract
            assert abs(got - want) <= 1e-12 * want, (got, want)  # what the kernel is built for


def test_ranges_accumulate_to_full_and_are_deterministic(layout):
    rng = np.random.default_rng(3)
    g = (rng.standard_normal(NBLK * 16384) * 0.1).astype(np.float32)
    dg = torch.from_numpy(g).cuda()
    full, _, _, _ = _norm(layout, dg, 0, NBLK)
    again, _, _, _ = _norm(layout, dg, 0, NBLK)
    assert full == again  # bit-identical
    s = torch.zeros(1, dtype=torch.float64, device="cuda")
    f = torch.zeros(1, dtype=torch.int32, device="cuda")
    for r in range(4):
        b0, b1 = F.fp8z1_shard_range(layout, r)
        F.fp8z1_grad_norm(layout, dg[b0 * 16384:], b0, b1, s, f)
    torch.cuda.synchronize()
    want = oracle.sumsq(g)[0]
    assert abs(s.item() - want) <= 1e-12 * want
    # a missing rank's partial is visible
    s2 = torch.zeros(1, dtype=torch.float64, device="cuda")
    for r in range(3):
        b0, b1 = F.fp8z1_shard_range(layout, r)
        F.fp8z1_grad_norm(layout, dg[b0 * 16384:], b0, b1, s2, f)
    torch.cuda.synchronize()
    assert abs(s2.item() - want) > 1e-3 * want


@pytest.mark.parametrize("fill", [1.0, 0.0])
@pytest.mark.parametrize("bad", [float("inf"), float("-inf"), float("nan"), -float("nan")])
@pytest.mark.parametrize("where", [0, 5 * 16384 + 77, 5 * 16384 + 8192 + 2, NBLK * 16384 - 1])
def test_found_inf(layout, bad, where, fill):
    # A nan leaves the running float sum of squares finite (max / min drop it)
    # and shows only in its low part; next to zeros the sum stays 0.  Both must
    # still send the unit to the double path, which raises the flag.
    g = np.full(NBLK * 16384, fill, np.float32)
    g[where] = bad
    dg = torch.from_numpy(g).cuda()
    _, found, _, _ = _norm(layout, dg, 0, NBLK)
    assert found == 1
    blk = where // 16384
    other = (blk + 1) % NBLK
    _, found, _, _ = _norm(layout, dg, other, other + 1)
    assert found == 0


def test_big_finite_not_flagged(layout):
    g = np.full(NBLK * 16384, 3e38, np.float32)
    got, found, _, _ = _norm(layout, torch.from_numpy(g).cuda(), 0, NBLK)
    assert found == 0
    want = oracle.sumsq(g)[0]
    assert abs(got - want) <= 1e-12 * want


def test_empty_range_changes_nothing(layout):
    s = torch.full((1,), 5.0, dtype=torch.float64, device="cuda")
    f = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = torch.ones(NBLK * 16384, device="cuda")
    F.fp8z1_grad_norm(layout, g, 4, 4, s, f)
    torch.cuda.synchronize()
    assert s.item() == 5.0 and f.item() == 0
