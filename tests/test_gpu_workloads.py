"""GPU parity on the workloads at their full sizes, through the C-ABI: the
unfused entry points (fold all grads -> per-rank norm partials summed ->
step on the rank's range -> unfold the codes) on every workload, and the MoE
buffer in the loop bench.py times (fused, steps enqueued ahead of their
found_inf), with a check of every block against the quantiser's definition.

The oracle checks every step on a seeded sample of blocks, one block at a
time: blocks are independent given the global scalars ("面向 Blockwise FP8
量化的 ZeRO 优化器设计" §总结: the update is elementwise), and the global sum
of squares is computed exactly by the oracle over every grad of every rank.
The oracle takes each sampled block's source tile from the oracle's own
lookup table and folds it itself.

Bars: fold / unfold bit-exact; norm within 1e-5 (and 1e-12 as built);
master / m / v / scales within 1e-6 relative; codes within one step on at
most 1e-4 of the sampled elements."""
import numpy as np
import pytest
import torch

import oracle
from blockwise_fp8_zero_fold_gb300 import fp8z1 as F
from blockwise_fp8_zero_fold_gb300 import synth
from blockwise_fp8_zero_fold_gb300.optimizer import shard_scale_view
from tests._gpu import assert_codes, assert_rel, lib, to_host  # noqa: F401

pytestmark = pytest.mark.gpu
B = 16384


class Harness:
    def __init__(self, w: synth.Workload, rank: int, n_sample: int, must=()):
        self.w = w
        self.dev = torch.device("cuda")
        self.L = F.fp8z1_build_layout(w.shapes, w.dp)
        self.nblk = F.fp8z1_layout_info(self.L)[0]
        self.b0, self.b1 = F.fp8z1_shard_range(self.L, rank)
        assert (self.b0, self.b1) == oracle.shard_range(self.nblk, w.dp, rank)
        self.lut = oracle.build_lut(w.shapes)
        nb = self.b1 - self.b0
        f32 = dict(dtype=torch.float32, device=self.dev)
        self.master = torch.empty(nb * B, **f32)
        self.m = torch.empty(nb * B, **f32)
        self.v = torch.empty(nb * B, **f32)
        self.codes = torch.full((nb * B,), 0xEE, dtype=torch.uint8, device=self.dev)
        self.scales = torch.full((nb,), -1.0, **f32)
        self.grad = torch.empty(self.nblk * B, **f32)  # every rank's folded grads
        self.sumsq = torch.zeros(1, dtype=torch.float64, device=self.dev)
        self.found = torch.zeros(1, dtype=torch.int32, device=self.dev)
        self.fp8 = [torch.full(s, 0xEE, dtype=torch.uint8, device=self.dev) for s in w.shapes]
        self.fp8_ptrs = F.param_pointers(self.fp8)
        self.scaler = F.fp8z1_loss_scaler(w.loss_scale, 0, 0, w.growth_interval)
        self.oscaler = oracle.Scaler(w.loss_scale, w.growth_interval)
        self.views_checked = 0

        rng = np.random.default_rng(1234 + rank)
        pick = set(int(x) for x in rng.choice(np.arange(self.b0, self.b1), min(n_sample, nb), replace=False))
        starts = np.cumsum([0] + [oracle.count_blocks([s]) for s in w.shapes])
        for a, b in zip(starts[:-1], starts[1:]):
            for k in (a, b - 1):
                if self.b0 <= k < self.b1:
                    pick.add(int(k))
        pick |= {int(k) for k in must if self.b0 <= k < self.b1}
        self.sample = np.array(sorted(pick), dtype=np.int64)
        self.local = torch.from_numpy(self.sample - self.b0).to(self.dev)

        # initial state: row-major on the device, folded by the library; the
        # oracle folds the sampled tiles itself
        self.state = {}
        for kind, buf in (("master", self.master), ("m", self.m), ("v", self.v)):
            rm = synth.make_state(w, kind, self.dev)
            F.fp8z1_fold(self.L, F.param_pointers(rm), buf, 4, self.b0, self.b1)
            self.state[kind] = np.stack([self.oracle_block(rm, k) for k in self.sample])
            del rm
        torch.cuda.synchronize()
        assert F.fp8z1_device_status(self.L) == 0

    def tile(self, rm, k):
        p, e, rb, cb, rr, cr = (int(x) for x in self.lut[k])
        return rm[p][e, 128 * rb:128 * rb + rr, 128 * cb:128 * cb + cr]

    def oracle_block(self, rm, k):
        t = np.ascontiguousarray(to_host(self.tile(rm, k)))
        return oracle.fold([(1,) + t.shape], [t.reshape((1,) + t.shape)])

    def check_scale_views(self, want):
        """The per-param scale views (the scales "unfolded" to [E, R/128,
        C/128], §总结) hold, at the (p, e, rb, cb) the oracle's table gives
        each sampled block, the oracle's scale of that block; a param with no
        expert wholly in the shard has no view."""
        views, wholes = {}, {}
        for i, k in enumerate(self.sample):
            p, e, rb, cb = (int(x) for x in self.lut[k][:4])
            if p not in views:
                views[p] = shard_scale_view(self.L, self.scales, self.b0, self.b1, p)
                mine = np.flatnonzero(self.lut[:, 0] == p)
                ex = self.lut[mine, 1]
                wholes[p] = {ee for ee in range(int(ex.max()) + 1)
                             if ((mine[ex == ee] >= self.b0) & (mine[ex == ee] < self.b1)).all()}
            v = views[p]
            if e not in wholes[p]:
                assert v is None or not (v[0] <= e < v[0] + v[1].shape[0])
                continue
            e0, view = v
            assert float(view[e - e0, rb, cb]) == float(want[i]), (k, p, e, rb, cb)
            self.views_checked += 1

    def gather(self, buf, per_block=B):
        return to_host(buf.view(-1, per_block)[self.local]) if per_block > 1 else to_host(buf[self.local])

    def step(self, t: int):
        w = self.w
        grads = synth.make_grads(w, t, self.dev)
        # ---- GPU, through the C-ABI
        F.fp8z1_fold(self.L, F.param_pointers(grads), self.grad, 4, 0, self.nblk)
        self.sumsq.zero_()
        self.found.zero_()
        for r in range(w.dp):  # the per-rank partials of the all-reduce
            a, b = F.fp8z1_shard_range(self.L, r)
            F.fp8z1_grad_norm(self.L, self.grad[a * B:], a, b, self.sumsq, self.found)
        hp = F.make_hp(step=self.scaler.step + 1, loss_scale=self.scaler.scale, **{
            k: v for k, v in w.hp().items() if k != "loss_scale"})
        F.fp8z1_step(self.L, hp, self.grad[self.b0 * B:], self.master, self.m, self.v, self.codes,
                     self.scales, self.b0, self.b1, self.sumsq, self.found)
        F.fp8z1_unfold(self.L, self.codes, self.fp8_ptrs, 1, self.b0, self.b1)
        found = int(self.found.item())
        F.fp8z1_scaler_update(self.scaler, found)

        # ---- oracle
        host_grads = [to_host(g) for g in grads]
        s_exact, f_exact = oracle.sumsq_parallel(host_grads, threads=16)
        assert found == f_exact
        if not f_exact:
            got = float(self.sumsq.item())
            assert abs(got - s_exact) <= 1e-5 * s_exact
            assert abs(got - s_exact) <= 1e-12 * s_exact, (got, s_exact)
        ohp = oracle.make_hp(step=self.oscaler.step + 1, loss_scale=self.oscaler.scale, **{
            k: v for k, v in w.hp().items() if k != "loss_scale"})
        g_blocks = np.stack([self.oracle_block(grads, k) for k in self.sample])
        assert np.array_equal(self.gather(self.grad[self.b0 * B:]).view(np.uint32),
                              g_blocks.view(np.uint32)), "folded grads differ"
        q = np.empty_like(g_blocks, dtype=np.uint8)
        s = np.empty(len(self.sample), np.float32)
        for i in range(len(self.sample)):
            qi, si, skipped = oracle.step(ohp, s_exact, f_exact, g_blocks[i], self.state["master"][i],
                                          self.state["m"][i], self.state["v"][i])
            assert skipped == bool(f_exact)
            if not skipped:
                q[i], s[i] = qi, si[0]
        self.oscaler.update(f_exact)
        assert (self.scaler.scale, self.scaler.step) == (self.oscaler.scale, self.oscaler.step)

        assert_rel(self.gather(self.master), self.state["master"], 1e-6, "master")
        assert_rel(self.gather(self.m), self.state["m"], 1e-6, "m")
        assert_rel(self.gather(self.v), self.state["v"], 1e-6, "v")
        exact = (np.array_equal(self.gather(self.master).view(np.uint32), self.state["master"].view(np.uint32))
                 and np.array_equal(self.gather(self.m).view(np.uint32), self.state["m"].view(np.uint32)))
        if not f_exact:
            gs = self.gather(self.scales, per_block=1)
            assert_rel(gs, s, 1e-6, "scales")
            self.check_scale_views(s)
            gq = self.gather(self.codes)
            frac = assert_codes(gq, q, "codes")
            exact = exact and frac == 0.0 and np.array_equal(gs, s)
            # the unfolded FP8 weights: the oracle unfolds its own codes of each sampled block
            for i, k in enumerate(self.sample):
                p, e, rb, cb, rr, cr = (int(x) for x in self.lut[k])
                want = np.zeros((1, rr, cr), np.uint8)
                oracle.unfold([(1, rr, cr)], q[i], [want])
                got = to_host(self.tile(self.fp8, k))
                d = np.abs(np.where(got & 0x80, -(got & 0x7F).astype(int), (got & 0x7F).astype(int))
                           - np.where(want[0] & 0x80, -(want[0] & 0x7F).astype(int), (want[0] & 0x7F).astype(int)))
                assert d.max() <= 1
        del grads, host_grads
        return found, exact


def _run(w, rank, steps, n_sample, must=()):
    h = Harness(w, rank, n_sample, must)
    out = [h.step(t) for t in range(1, steps + 1)]
    assert F.fp8z1_device_status(h.L) == 0
    return h, out


@pytest.mark.parametrize("rank", [0, 1])
def test_tiny_all_blocks(lib, rank):
    w = synth.workload("tiny")
    h, out = _run(w, rank, w.steps, n_sample=10)
    assert len(h.sample) == 3 and [f for f, _ in out] == [0, 0, 0]
    assert all(e for _, e in out)
    assert h.views_checked == 0  # each rank holds half of the one weight: no view


def test_dense_ten_steps(lib):
    w = synth.workload("dense")
    h, out = _run(w, 0, w.steps, n_sample=160)
    assert all(f == 0 for f, _ in out) and all(e for _, e in out)
    assert h.views_checked == len(h.sample) * w.steps


def test_tiny_whole_weight_scale_view(lib):
    w = synth.workload("tiny", dp=1, rank=0)
    h, out = _run(w, 0, w.steps, n_sample=10)
    assert len(h.sample) == 6 and h.views_checked == 6 * w.steps


def test_moe_rank3_of_8(lib):
    w = synth.workload("moe")
    h, out = _run(w, 3, w.steps, n_sample=160)
    assert (h.b0, h.b1) == (32256, 43008)
    assert all(f == 0 for f, _ in out) and all(e for _, e in out)
    # the shard holds experts 18-23 of gate_up whole: their scale view
    assert h.views_checked == len(h.sample) * w.steps
    e0, view = shard_scale_view(h.L, h.scales, h.b0, h.b1, 0)
    assert e0 == 18 and tuple(view.shape) == (6, 56, 32)
    assert shard_scale_view(h.L, h.scales, h.b0, h.b1, 1) is None


def test_moe_full_buffer_with_zero_blocks(lib):
    w = synth.workload("moe", dp=1, rank=0)
    # a few of the all-zero tiles must be in the sample: they keep scale 1
    tiles = synth.zero_tiles(w)
    gu = oracle.count_blocks([w.shapes[0]])
    rb0, cb0 = -(-w.shapes[0][1] // 128), -(-w.shapes[0][2] // 128)
    rb1, cb1 = -(-w.shapes[1][1] // 128), -(-w.shapes[1][2] // 128)
    must = [int((e * rb0 + a) * cb0 + b) for e, a, b in tiles[0][:4].tolist()]
    must += [gu + int((e * rb1 + a) * cb1 + b) for e, a, b in tiles[1][:4].tolist()]
    h, out = _run(w, 0, 2, n_sample=160, must=must)
    assert all(f == 0 for f, _ in out) and all(e for _, e in out)
    idx = [int(np.flatnonzero(h.sample == k)[0]) for k in must]
    gs = h.gather(h.scales, per_block=1)
    assert (gs[idx] == 1.0).all()
    assert (h.gather(h.codes)[idx] == 0).all()


def test_ragged_skip_step(lib):
    w = synth.workload("ragged")
    starts = np.cumsum([0] + [oracle.count_blocks([s]) for s in w.shapes])
    must = list(range(int(starts[w.inf_param]), int(starts[w.inf_param + 1])))
    h, out = _run(w, 0, w.steps, n_sample=240, must=must)
    assert [f for f, _ in out] == [0, 1, 0]
    assert all(e for _, e in out)
    assert h.views_checked == len(h.sample) * 2  # the two steps not skipped
    # S halves on the skipped step and t does not advance
    assert (h.scaler.scale, h.scaler.step) == (32768.0, 2)


def test_large_two_steps_and_bf16_fold(lib):
    w = synth.workload("large")
    h, out = _run(w, 0, 2, n_sample=120)
    assert all(f == 0 for f, _ in out) and all(e for _, e in out)
    # bf16 fold / unfold of the same weights (2-byte elements)
    rm = synth.make_state(w, "master", h.dev)
    bf = [t.to(torch.bfloat16) for t in rm]
    del rm
    buf = torch.empty(h.nblk * B, dtype=torch.bfloat16, device=h.dev)
    F.fp8z1_fold(h.L, F.param_pointers(bf), buf, 2, 0, h.nblk)
    for k in h.sample[:40]:
        t = to_host(h.tile([x.view(torch.int16) for x in bf], int(k)))
        want = oracle.fold([(1,) + t.shape], [np.ascontiguousarray(t).reshape((1,) + t.shape)])
        assert np.array_equal(to_host(buf.view(torch.int16)[int(k) * B:(int(k) + 1) * B]), want)
    back = [torch.zeros_like(x) for x in bf]
    F.fp8z1_unfold(h.L, buf, F.param_pointers(back), 2, 0, h.nblk)
    torch.cuda.synchronize()
    for a, b in zip(bf, back):  # unfold(fold(x)) == x over every element
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("name", ["moe", "ragged", "dense"])
def test_bench_loop_every_block(lib, name):
    """A workload's whole buffer in exactly the loop bench.py times (MoE: the
    bench's default; ragged: the padding-aware step kernel on partial blocks;
    dense: both kernels, full-tile runs and a padded param): ShardOptimizer on the
    fused path, steps enqueued ahead of their found_inf (launch_step_async),
    the same grads every step.  After three steps: sampled blocks against the
    oracle (master / m / v / scales bit-exact, the row-major FP8 tiles), the
    norm against the exact sum, and on every block of the buffer the
    quantiser's definition ("面向 Blockwise FP8 量化的 ZeRO 优化器设计" §总结):
    scale = amax/448 (1 when amax = 0) of the new FP32 master, codes = the
    E4M3 round-to-nearest-even of master/scale (torch.float8_e4m3fn casts)."""
    from blockwise_fp8_zero_fold_gb300.optimizer import ShardOptimizer
    w = synth.workload(name, dp=1, rank=0)
    dev = torch.device("cuda")
    opt = ShardOptimizer(w.shapes, loss_scale=w.loss_scale, growth_interval=w.growth_interval,
                         **{k: v for k, v in w.hp().items() if k != "loss_scale"})
    lut = oracle.build_lut(w.shapes)
    rng = np.random.default_rng(77)
    tiles = synth.zero_tiles(w)
    cb0 = -(-w.shapes[0][2] // 128)
    rb0 = -(-w.shapes[0][1] // 128)
    sample = sorted(set(int(x) for x in rng.choice(opt.nblk, 120, replace=False))
                    | {0, opt.nblk - 1} | {int((e * rb0 + a) * cb0 + b) for e, a, b in tiles[0][:3].tolist()})

    def tile(rm, k):
        p, e, rb, cb, rr, cr = (int(x) for x in lut[k])
        return rm[p][e, 128 * rb:128 * rb + rr, 128 * cb:128 * cb + cr]

    def oblock(rm, k):
        t = np.ascontiguousarray(to_host(tile(rm, k)))
        return oracle.fold([(1,) + t.shape], [t.reshape((1,) + t.shape)])

    state = {}
    for kind in ("master", "m", "v"):
        rm = synth.make_state(w, kind, dev)
        opt.fold_into(rm, getattr(opt, kind))
        state[kind] = [oblock(rm, k) for k in sample]
        del rm
    grads = synth.make_grads(w, 1, dev)
    fp8 = [torch.full(s, 0x7F, dtype=torch.uint8, device=dev) for s in w.shapes]
    found = []
    for _ in range(3):
        found += opt.launch_step_async(grads, fp8)
    found += opt.drain()
    assert found == [0, 0, 0] and opt.scaler.step == 3

    exact, fi = oracle.sumsq_parallel([to_host(g) for g in grads], threads=16)
    assert fi == 0 and abs(float(opt.sumsq.item()) - exact) <= 1e-12 * exact
    views = opt.scale_views()  # the whole buffer: every param has its view
    assert all(v is not None and tuple(v.shape) == (e, -(-r // 128), -(-c // 128))
               for v, (e, r, c) in zip(views, w.shapes))
    for i, k in enumerate(sample):
        g = oblock(grads, k)
        for t in range(1, 4):
            q, sc, _ = oracle.step(oracle.make_hp(step=t, **w.hp()), exact, 0, g, state["master"][i],
                                   state["m"][i], state["v"][i])
        for name in ("master", "m", "v"):
            got = to_host(getattr(opt, name)[k * B:(k + 1) * B])
            assert np.array_equal(got.view(np.uint32), state[name][i].view(np.uint32)), (name, k)
        assert float(opt.scales[k]) == float(sc[0])
        p, e, rb, cb, rr, cr = (int(x) for x in lut[k])
        assert float(views[p][e, rb, cb]) == float(sc[0]), k
        want = np.zeros((1, rr, cr), np.uint8)
        oracle.unfold([(1, rr, cr)], q, [want])
        assert np.array_equal(to_host(tile(fp8, k)), want[0]), k

    # every block: the scale and the codes from their definitions
    master = opt.master.view(opt.nblk, B)
    amax = master.abs().amax(dim=1)
    # a tensor divisor: torch divides by a Python scalar through its reciprocal,
    # which can be an ulp off the IEEE quotient the definition asks for
    want_scale = torch.where(amax == 0, torch.ones_like(amax), amax / torch.full_like(amax, 448.0))
    assert torch.equal(opt.scales.view(torch.int32), want_scale.view(torch.int32))
    folded = torch.empty(opt.nblk * B, dtype=torch.uint8, device=dev)
    F.fp8z1_fold(opt.layout, F.param_pointers(fp8), folded, 1, 0, opt.nblk)
    want_codes = (master / want_scale[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).view(-1)
    assert torch.equal(folded, want_codes)
    assert (opt.scales == 1.0).sum().item() >= len(tiles[0]) + len(tiles[1])  # the all-zero tiles
    assert F.fp8z1_device_status(opt.layout) == 0
