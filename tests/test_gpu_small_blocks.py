"""GPU parity of the fused step on layouts made of small and partial blocks
("面向 Blockwise FP8 量化的 ZeRO 优化器设计" §块粒度切分: padding to multiples
of 128 leaves partial blocks on every weight whose R or C is not one): forty
one-block weights, one-row and one-column weights, C < 4 and every C % 4, real
columns and rows on either side of each point where a warp starts taking
several rows of a narrow block, weights whose storage starts 1-3 elements into
a buffer, full tiles among the partial ones, a 512-block full-tile run between
padded weights, the three scalar forms, a skipped step and an unreadable
param.

Every case is compared with the oracle -- master / m / v / scales bit for
bit, the row-major codes byte for byte, every code outside the real elements
of the range untouched -- and the whole buffer with the same buffer stepped as
two ranges."""
import numpy as np
import pytest
import torch

import oracle
from blockwise_fp8_zero_fold_gb300 import fp8z1 as F
from tests._gpu import lib, to_host  # noqa: F401

pytestmark = pytest.mark.gpu
B = 16384
SENTINEL = 0x7F  # an E4M3 NaN code, which the step never writes

CASES = {
    # 40 tiny weights: units of eight blocks
    "tiny_many": [(1, int(r), int(c)) for r, c in zip(range(1, 41), range(41, 1, -1))],
    "narrow_and_flat": [(1, 300, 1), (1, 1, 300), (2, 129, 3), (1, 5, 2), (3, 1, 1), (1, 700, 6)],
    "ragged_mix": [(1, 17, 690), (2, 255, 3), (3, 129, 257), (1, 1000, 131), (1, 128, 384), (2, 200, 130)],
    "every_c_mod_4": [(1, 150 + k, 260 + k) for k in range(8)],
    # real columns on either side of every warp-row split (a warp takes 32 / W rows
    # of a block whose real chunks a row fit in W = 16, 8, 4, 2, 1), rows on either
    # side of a task and of a warp's share
    "row_split_edges": [(1, r, c) for c in (4, 5, 8, 9, 16, 17, 32, 33, 64, 65, 127, 129)
                        for r in (1, 31, 33, 97, 130)],
}


def _hp(step=2, loss_scale=1024.0, max_norm=0.5):
    return dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=max_norm,
                loss_scale=loss_scale, step=step)


class Case:
    """Row-major grads and FP8 weights on the device, each param's storage
    starting `skew[i]` elements into its own buffer (the grads 4-byte aligned,
    the rows not 16-byte aligned), and the oracle's folded state."""

    def __init__(self, shapes, seed, skew=False, dp=1):
        rng = np.random.default_rng(seed)
        self.shapes = shapes
        self.L = F.fp8z1_build_layout(shapes, dp_size=dp)
        self.nblk = F.fp8z1_layout_info(self.L)[0]
        self.gh = [(rng.standard_normal(s) * 1024e-3).astype(np.float32) for s in shapes]
        self.ph = [(rng.standard_normal(s) * 0.02).astype(np.float32) for s in shapes]
        self.mh = [(rng.standard_normal(s) * 1e-4).astype(np.float32) for s in shapes]
        self.vh = [np.abs(rng.standard_normal(s) * 1e-8).astype(np.float32) for s in shapes]
        self.skew = [int(rng.integers(0, 4)) if skew else 0 for _ in shapes]
        self.gbuf, self.dg = [], []
        for x, k in zip(self.gh, self.skew):
            buf = torch.zeros(x.size + 4, dtype=torch.float32, device="cuda")
            buf[k:k + x.size] = torch.from_numpy(x.reshape(-1)).cuda()
            self.gbuf.append(buf)
            self.dg.append(buf[k:k + x.size].view(x.shape))
        self.gptrs = F.param_pointers(self.dg)
        self.og = oracle.fold(shapes, self.gh)
        self.exact, self.of = oracle.sumsq(self.og)

    def sums(self, found=0):
        s = torch.tensor([self.exact], dtype=torch.float64, device="cuda")
        f = torch.tensor([found], dtype=torch.int32, device="cuda")
        return s, f

    def state(self, b0, b1):
        sl = slice(b0 * B, b1 * B)
        op, om, ov = (oracle.fold(self.shapes, x)[sl].copy() for x in (self.ph, self.mh, self.vh))
        return op, om, ov

    def device_state(self, b0, b1):
        op, om, ov = self.state(b0, b1)
        return [torch.from_numpy(x.copy()).cuda() for x in (op, om, ov)]

    def fp8(self):
        """FP8 weights with a sentinel everywhere, 3 guard bytes past each."""
        bufs = [torch.full((x.size + 3 + k,), SENTINEL, dtype=torch.uint8, device="cuda")
                for x, k in zip(self.gh, self.skew)]
        views = [b[k:k + x.size].view(x.shape) for b, x, k in zip(bufs, self.gh, self.skew)]
        return bufs, views

    def step(self, b0, b1, hp, state, views, scales, form="value", found=0):
        s, f = self.sums(found)
        kw = dict(d_grad_params=self.gptrs, master_shard=state[0], m_shard=state[1], v_shard=state[2],
                  d_fp8_params=F.param_pointers(views), scale_shard=scales, b0=b0, b1=b1, d_sumsq=s,
                  d_found_inf=f)
        if form == "value":
            F.fp8z1_step_fused(self.L, F.make_hp(**hp), **kw)
        elif form == "select":
            other = dict(hp, step=hp["step"] + 5, loss_scale=hp["loss_scale"] * 2)
            sel = torch.ones(1, dtype=torch.int32, device="cuda")
            F.fp8z1_step_fused_select(self.L, F.make_hp(**other), F.make_hp(**hp), sel, **kw)
        else:
            h = F.fp8z1_step_scalars_from_hp(F.make_hp(**hp))
            d = torch.zeros(10, dtype=torch.float32, device="cuda")
            hpin = torch.from_numpy(np.frombuffer(bytes(h), dtype=np.float32).copy()).pin_memory()
            F.fp8z1_step_fused_dev(self.L, hpin, d, **kw)
        torch.cuda.synchronize()

    def oracle_step(self, b0, b1, hp):
        op, om, ov = self.state(b0, b1)
        q, sc, skipped = oracle.step(oracle.make_hp(**hp), self.exact, self.of,
                                     self.og[b0 * B:b1 * B].copy(), op, om, ov)
        assert not skipped
        want8 = [np.full(x.shape, SENTINEL, np.uint8) for x in self.gh]
        oracle.unfold(self.shapes, q, want8, b0, b1)
        return (op, om, ov), sc, want8

    def check(self, got_state, got_scales, bufs, want_state, want_scales, want8, what):
        for g, w, name in zip(got_state, want_state, ("master", "m", "v")):
            assert np.array_equal(to_host(g).view(np.uint32), w.view(np.uint32)), (what, name)
        assert np.array_equal(to_host(got_scales).view(np.uint32), want_scales.view(np.uint32)), (what, "scales")
        for i, (buf, x, k) in enumerate(zip(bufs, self.gh, self.skew)):
            got = to_host(buf)
            assert (got[:k] == SENTINEL).all() and (got[k + x.size:] == SENTINEL).all(), (what, "guard", i)
            assert np.array_equal(got[k:k + x.size].reshape(x.shape), want8[i]), (what, "codes", i)


def _run(case, b0, b1, hp, form="value"):
    st = case.device_state(b0, b1)
    sc = torch.full((b1 - b0,), -1.0, device="cuda")
    bufs, views = case.fp8()
    n0 = F.fp8z1_kernel_launches()
    case.step(b0, b1, hp, st, views, sc, form)
    return st, sc, bufs, F.fp8z1_kernel_launches() - n0


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("skew", [False, True])
def test_small_blocks_match_oracle(lib, name, skew):
    case = Case(CASES[name], seed=len(name) * 7 + skew, skew=skew)
    hp = _hp()
    want_state, want_sc, want8 = case.oracle_step(0, case.nblk, hp)
    # the whole buffer: one launch (no weight here is a 512-block full-tile run)
    st, sc, bufs, launches = _run(case, 0, case.nblk, hp)
    assert launches == 1
    case.check(st, sc, bufs, want_state, want_sc, want8, "whole buffer")
    # the same buffer stepped as two ranges: the same bytes
    cut = case.nblk // 2
    st2 = case.device_state(0, case.nblk)
    sc2 = torch.full((case.nblk,), -1.0, device="cuda")
    bufs2, views2 = case.fp8()
    for a, b in ((0, cut), (cut, case.nblk)):
        sub = [t[a * B:b * B] for t in st2]
        case.step(a, b, hp, sub, views2, sc2[a:b])
    case.check(st2, sc2, bufs2, want_state, want_sc, want8, "two ranges")
    assert F.fp8z1_device_status(case.L) == 0


@pytest.mark.parametrize("form", ["select", "device"])
def test_small_blocks_scalar_forms(lib, form):
    case = Case(CASES["ragged_mix"], seed=5, skew=True)
    hp = _hp(step=3)
    want_state, want_sc, want8 = case.oracle_step(0, case.nblk, hp)
    st, sc, bufs, launches = _run(case, 0, case.nblk, hp, form)
    assert launches == 1
    case.check(st, sc, bufs, want_state, want_sc, want8, form)


@pytest.mark.parametrize("dp", [2, 3])
def test_small_blocks_rank_ranges(lib, dp):
    # a full-tile run between padded weights: three launches per rank that holds all three
    shapes = CASES["tiny_many"] + [(1, 128 * 32, 128 * 16)] + CASES["ragged_mix"]
    case = Case(shapes, seed=11 + dp, dp=dp)
    hp = _hp(step=1)
    for r in range(dp):
        b0, b1 = F.fp8z1_shard_range(case.L, r)
        want_state, want_sc, want8 = case.oracle_step(b0, b1, hp)
        st, sc, bufs, _ = _run(case, b0, b1, hp)
        case.check(st, sc, bufs, want_state, want_sc, want8, f"rank {r}")


def test_small_blocks_skip_and_unreadable_param(lib):
    case = Case(CASES["ragged_mix"], seed=9)
    hp = _hp()
    # a skipped step writes nothing
    st = case.device_state(0, case.nblk)
    before = [to_host(t).copy() for t in st]
    sc = torch.full((case.nblk,), -1.0, device="cuda")
    bufs, views = case.fp8()
    case.step(0, case.nblk, hp, st, views, sc, found=1)
    for t, b in zip(st, before):
        assert np.array_equal(to_host(t).view(np.uint32), b.view(np.uint32))
    assert (to_host(sc) == -1.0).all()
    assert all((to_host(b) == SENTINEL).all() for b in bufs)
    # a null grad pointer: that weight's blocks are left untouched and reported
    want_state, want_sc, want8 = case.oracle_step(0, case.nblk, hp)
    saved = case.gptrs.clone()
    case.gptrs[3] = 0
    st = case.device_state(0, case.nblk)
    sc = torch.full((case.nblk,), -1.0, device="cuda")
    bufs, views = case.fp8()
    case.step(0, case.nblk, hp, st, views, sc)
    case.gptrs.copy_(saved)
    assert F.fp8z1_device_status(case.L) == F.DEVSTATUS_BADPTR
    starts = np.cumsum([0] + [oracle.count_blocks([s]) for s in case.shapes])
    a, b = int(starts[3]), int(starts[4])
    init = case.state(0, case.nblk)
    for i, name in enumerate(("master", "m", "v")):
        got = to_host(st[i])
        want = want_state[i].copy()
        want[a * B:b * B] = init[i][a * B:b * B]
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), name
    wsc = want_sc.copy()
    wsc[a:b] = -1.0
    assert np.array_equal(to_host(sc), wsc)
    for i, buf in enumerate(bufs):
        got = to_host(buf)[:case.gh[i].size].reshape(case.gh[i].shape)
        want = np.full_like(want8[i], SENTINEL) if i == 3 else want8[i]
        assert np.array_equal(got, want), i
