"""GPU parity: the fused unscale + clip + AdamW + quantise step against the
oracle on the same seeded inputs.

Bars: master / m / v / scales within 1e-6 relative (|want| = 0 -> equal);
E4M3 codes within one code step on at most 1e-4 of elements.  The kernel and
the oracle follow one FP32 operation order, so the expected difference is 0,
and the tests also report exact agreement."""
import numpy as np
import pytest
import torch

import oracle
from blockwise_fp8_zero_fold_gb300 import fp8z1 as F
from tests._gpu import assert_codes, assert_rel, lib, to_host  # noqa: F401

pytestmark = pytest.mark.gpu
B = 16384


def _hp(**kw):
    d = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=1.0,
             loss_scale=1024.0, step=1)
    d.update(kw)
    return d


class Shard:
    """One folded shard on the device and the same state on the host."""

    def __init__(self, nb, rng, master_sigma=0.02, m_sigma=0.0, v_sigma=0.0):
        n = nb * B
        self.nb = nb
        self.p = (rng.standard_normal(n) * master_sigma).astype(np.float32)
        self.m = (rng.standard_normal(n) * m_sigma).astype(np.float32)
        self.v = np.abs(rng.standard_normal(n) * v_sigma).astype(np.float32)
        self.dp = torch.from_numpy(self.p.copy()).cuda()
        self.dm = torch.from_numpy(self.m.copy()).cuda()
        self.dv = torch.from_numpy(self.v.copy()).cuda()
        self.dq = torch.full((n,), 0xEE, dtype=torch.uint8, device="cuda")
        self.ds = torch.full((nb,), -1.0, dtype=torch.float32, device="cuda")

    def gpu_step(self, L, hp, g, b0=0, sumsq=None, found=None):
        dg = torch.from_numpy(g).cuda()
        s = torch.zeros(1, dtype=torch.float64, device="cuda") if sumsq is None else sumsq
        f = torch.zeros(1, dtype=torch.int32, device="cuda") if found is None else found
        if sumsq is None:
            F.fp8z1_grad_norm(L, dg, b0, b0 + self.nb, s, f)
        F.fp8z1_step(L, F.make_hp(**hp), dg, self.dp, self.dm, self.dv, self.dq, self.ds,
                     b0, b0 + self.nb, s, f)
        torch.cuda.synchronize()

    def oracle_step(self, hp, g, sumsq=None, found=None):
        if sumsq is None:
            sumsq, found = oracle.sumsq(g)
        q, s, skipped = oracle.step(oracle.make_hp(**hp), sumsq, found, g, self.p, self.m, self.v)
        return q, s, skipped

    def compare(self, q, s, exact=True):
        gp, gm, gv = to_host(self.dp), to_host(self.dm), to_host(self.dv)
        assert_rel(gp, self.p, 1e-6, "master")
        assert_rel(gm, self.m, 1e-6, "m")
        assert_rel(gv, self.v, 1e-6, "v")
        gs, gq = to_host(self.ds), to_host(self.dq)
        assert_rel(gs, s, 1e-6, "scales")
        frac = assert_codes(gq, q, "codes")
        if exact:
            assert np.array_equal(gp.view(np.uint32), self.p.view(np.uint32))
            assert np.array_equal(gm.view(np.uint32), self.m.view(np.uint32))
            assert np.array_equal(gv.view(np.uint32), self.v.view(np.uint32))
            assert np.array_equal(gs, s)
            assert frac == 0.0


@pytest.mark.parametrize("case", ["no_clip", "clip", "clip_S65536", "moments", "wd0"])
def test_multi_step_parity(lib, case):
    rng = np.random.default_rng(hash(case) % 2**32)
    nb = 7
    L = F.fp8z1_build_layout([(nb, 128, 128)])
    kw = dict(m_sigma=1e-4, v_sigma=1e-8) if case == "moments" else {}
    sh = Shard(nb, rng, **kw)
    S = 65536.0 if case == "clip_S65536" else 1024.0
    max_norm = {"no_clip": 1e9, "clip": 0.05, "clip_S65536": 0.8}.get(case, 1.0)
    wd = 0.0 if case == "wd0" else 0.1
    for t in range(1, 4):
        g = (rng.standard_normal(nb * B) * 1e-3 * S).astype(np.float32)
        hp = _hp(step=t, loss_scale=S, max_norm=max_norm, weight_decay=wd)
        sh.gpu_step(L, hp, g)
        q, s, skipped = sh.oracle_step(hp, g)
        assert not skipped
        sh.compare(q, s)


def test_quantiser_sweep_exact_values(lib):
    """lr = 0, wd = 0 and zero grads leave p unchanged, so the codes are the
    E4M3 codes of chosen values: with amax = 448 the scale is exactly 1."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float64)
    pos = np.unique(np.abs(vals))
    mids = (pos[:-1] + pos[1:]) / 2
    x = np.concatenate([pos, mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                        np.nextafter(mids.astype(np.float32), np.float32(1000)),
                        [2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -11, 1e-30, 0.0]]).astype(np.float32)
    x = np.concatenate([x, -x])
    rng = np.random.default_rng(0)
    blk1 = np.zeros(B, np.float32)
    blk1[:x.size] = x
    blk1[x.size:] = rng.uniform(-448, 448, B - x.size).astype(np.float32)
    blk1[-1] = 448.0
    blk2 = (rng.standard_normal(B) * 3e-3).astype(np.float32)  # a scale that is not 1
    blk3 = np.zeros(B, np.float32)                              # amax 0 -> scale 1
    blk3[::5] = -0.0
    L = F.fp8z1_build_layout([(3, 128, 128)])
    sh = Shard(3, rng)
    sh.p = np.concatenate([blk1, blk2, blk3])
    sh.dp.copy_(torch.from_numpy(sh.p))
    hp = _hp(lr=0.0, weight_decay=0.0)
    g = np.zeros(3 * B, np.float32)
    sh.gpu_step(L, hp, g)
    q, s, _ = sh.oracle_step(hp, g)
    assert s[0] == 1.0 and s[2] == 1.0
    sh.compare(q, s)


def test_skip_step_writes_nothing(lib):
    rng = np.random.default_rng(9)
    nb = 4
    L = F.fp8z1_build_layout([(nb, 128, 128)])
    sh = Shard(nb, rng, m_sigma=1e-4, v_sigma=1e-8)
    before = [to_host(t).copy() for t in (sh.dp, sh.dm, sh.dv, sh.dq, sh.ds)]
    g = (rng.standard_normal(nb * B) * 1.0).astype(np.float32)
    g[3 * B + 11] = np.inf
    sh.gpu_step(L, _hp(), g)
    after = [to_host(t) for t in (sh.dp, sh.dm, sh.dv, sh.dq, sh.ds)]
    for a, b in zip(before, after):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    q, s, skipped = sh.oracle_step(_hp(), g)
    assert skipped


def test_subrange_writes_only_its_blocks_and_matches_split_ranks(lib):
    """DP = 3 simulated ranks on one buffer: the global norm is the sum of the
    three range partials, each rank steps its range; together they equal one
    whole-buffer step bit for bit."""
    rng = np.random.default_rng(10)
    nb = 8
    L = F.fp8z1_build_layout([(2, 512, 128)], dp_size=3)
    assert F.fp8z1_layout_info(L)[0] == nb
    whole = Shard(nb, rng, m_sigma=1e-4, v_sigma=1e-8)
    split = Shard(nb, np.random.default_rng(10), m_sigma=1e-4, v_sigma=1e-8)
    g = (rng.standard_normal(nb * B) * 1e-3 * 1024).astype(np.float32)
    hp = _hp(max_norm=0.5)
    whole.gpu_step(L, hp, g)
    dg = torch.from_numpy(g).cuda()
    s = torch.zeros(1, dtype=torch.float64, device="cuda")
    f = torch.zeros(1, dtype=torch.int32, device="cuda")
    for r in range(3):
        b0, b1 = F.fp8z1_shard_range(L, r)
        F.fp8z1_grad_norm(L, dg[b0 * B:], b0, b1, s, f)
    for r in range(3):
        b0, b1 = F.fp8z1_shard_range(L, r)
        F.fp8z1_step(L, F.make_hp(**hp), dg[b0 * B:], split.dp[b0 * B:], split.dm[b0 * B:],
                     split.dv[b0 * B:], split.dq[b0 * B:], split.ds[b0:], b0, b1, s, f)
    torch.cuda.synchronize()
    for a, b in [(whole.dp, split.dp), (whole.dm, split.dm), (whole.dv, split.dv),
                 (whole.dq, split.dq), (whole.ds, split.ds)]:
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    # the oracle on the same inputs
    q, sc, _ = whole.oracle_step(hp, g)
    whole.compare(q, sc)
    # a range step leaves the other blocks untouched
    third = Shard(nb, np.random.default_rng(11))
    before = to_host(third.dp).copy()
    F.fp8z1_step(L, F.make_hp(**hp), dg[3 * B:], third.dp[3 * B:], third.dm[3 * B:], third.dv[3 * B:],
                 third.dq[3 * B:], third.ds[3:], 3, 6, s, f)
    torch.cuda.synchronize()
    got = to_host(third.dp)
    assert np.array_equal(got[:3 * B], before[:3 * B]) and np.array_equal(got[6 * B:], before[6 * B:])
    assert (to_host(third.dq)[:3 * B] == 0xEE).all() and (to_host(third.ds)[6:] == -1.0).all()
