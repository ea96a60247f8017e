"""GPU parity on the ragged workload as its configuration states it literally:
4000 2-D weights with R and C uniform in [17, 3000] (9.08 G real elements,
602268 blocks, 9.87 G padded elements, offsets past 2^33), through the fused
path the bench times (fp8z1_fold_norm from the row-major grads, then
fp8z1_step_fused reading the grads through the block table and writing the
codes row-major), three steps with +inf in one weight on step 2.

"面向 Blockwise FP8 量化的 ZeRO 优化器设计" §块粒度切分: every quantised dim is
padded to a multiple of 128 and the table records the real extent, which
here leaves most weights with partial blocks on two edges.

Checks, through the C-ABI:
- the norm against the oracle's exact sum over every grad (1e-12 as built;
  the bar is 1e-5) and the inf flag of step 2 (the skipped step: state
  unchanged, S halved, t not advanced -- "DeepSpeed ZeRO 优化" §六);
- a seeded sample of blocks (every block of the weight with the inf among
  them) against the oracle's step, bit for bit on master / m / v / scales and
  on the row-major FP8 tiles;
- every block of the buffer against the quantiser's definition (§总结):
  scale = amax/448 (1 when amax = 0) of the new FP32 master, codes = the
  E4M3 round-to-nearest-even of master / scale."""
import numpy as np
import pytest
import torch

import oracle
from blockwise_fp8_zero_fold_gb300 import fp8z1 as F
from blockwise_fp8_zero_fold_gb300 import synth
from tests._gpu import lib, to_host  # noqa: F401

pytestmark = pytest.mark.gpu
B = 16384


def test_ragged_literal_three_fused_steps(lib):
    from blockwise_fp8_zero_fold_gb300.optimizer import ShardOptimizer
    torch.cuda.empty_cache()
    w = synth.workload("ragged_literal")
    dev = torch.device("cuda")
    opt = ShardOptimizer(w.shapes, loss_scale=w.loss_scale, growth_interval=w.growth_interval,
                         **{k: v for k, v in w.hp().items() if k != "loss_scale"})
    assert opt.nblk == oracle.count_blocks(w.shapes) == 602268
    assert opt.n_real == w.n_real and opt.n_padded > 2 ** 33
    lut = oracle.build_lut(w.shapes)

    starts = np.cumsum([0] + [oracle.count_blocks([s]) for s in w.shapes])
    rng = np.random.default_rng(2026)
    sample = set(int(x) for x in rng.choice(opt.nblk, 200, replace=False))
    sample |= set(range(int(starts[w.inf_param]), int(starts[w.inf_param + 1])))
    sample |= {0, opt.nblk - 1, int(starts[-2])}
    sample = sorted(sample)

    def tile(rm, k):
        p, e, rb, cb, rr, cr = (int(x) for x in lut[k])
        return rm[p][e, 128 * rb:128 * rb + rr, 128 * cb:128 * cb + cr]

    def oblock(rm, k):
        t = np.ascontiguousarray(to_host(tile(rm, k)))
        return oracle.fold([(1,) + t.shape], [t.reshape((1,) + t.shape)])

    # initial state: master drawn row-major and folded by the library; the
    # workload's moments start at zero, as the optimizer's buffers do
    assert w.m_sigma == 0.0 and w.v_sigma == 0.0
    rm = synth.make_state(w, "master", dev)
    opt.fold_into(rm, opt.master)
    state = {"master": [oblock(rm, k) for k in sample],
             "m": [np.zeros(B, np.float32) for _ in sample],
             "v": [np.zeros(B, np.float32) for _ in sample]}
    del rm
    torch.cuda.empty_cache()

    grads = synth.make_grads(w, 1, dev)
    fp8 = [torch.full(s, 0x7F, dtype=torch.uint8, device=dev) for s in w.shapes]
    gptrs, fptrs = opt.pointers(grads), opt.pointers(fp8)
    oscaler = oracle.Scaler(w.loss_scale, w.growth_interval)
    want_scale = [None] * len(sample)
    want_codes = [None] * len(sample)
    for t in range(1, 4):
        if t > 1:
            synth.make_grads(w, t, dev, out=grads)
        found = opt.step(gptrs, fptrs)
        # the oracle: exact norm over every grad, then each sampled block
        exact, f_exact = oracle.sumsq_parallel([to_host(g) for g in grads], threads=16)
        assert found == f_exact == (1 if t == w.inf_step else 0)
        if not f_exact:
            got = float(opt.sumsq.item())
            assert abs(got - exact) <= 1e-5 * exact
            assert abs(got - exact) <= 1e-12 * exact, (got, exact)
        hp = oracle.make_hp(step=oscaler.step + 1, loss_scale=oscaler.scale,
                            **{k: v for k, v in w.hp().items() if k != "loss_scale"})
        for i, k in enumerate(sample):
            g = oblock(grads, k)
            q, s, skipped = oracle.step(hp, exact, f_exact, g, state["master"][i], state["m"][i], state["v"][i])
            assert skipped == bool(f_exact)
            if not skipped:
                want_scale[i], want_codes[i] = float(s[0]), q
        oscaler.update(f_exact)
        assert (opt.scaler.scale, opt.scaler.step) == (oscaler.scale, oscaler.step)
        for i, k in enumerate(sample):
            for name in ("master", "m", "v"):
                got = to_host(getattr(opt, name)[k * B:(k + 1) * B])
                assert np.array_equal(got.view(np.uint32), state[name][i].view(np.uint32)), (t, name, k)
            assert float(opt.scales[k]) == want_scale[i], (t, k)
            p, e, rb, cb, rr, cr = (int(x) for x in lut[k])
            want = np.zeros((1, rr, cr), np.uint8)
            oracle.unfold([(1, rr, cr)], want_codes[i], [want])
            assert np.array_equal(to_host(tile(fp8, k)), want[0]), (t, k)
    assert (opt.scaler.scale, opt.scaler.step) == (32768.0, 2)
    assert F.fp8z1_device_status(opt.layout) == 0

    # every block: the scale and the codes from their definitions, in chunks
    # (the folded code buffer the fused path leaves unused takes the fold of
    # the row-major FP8 weights)
    F.fp8z1_fold(opt.layout, fptrs, opt.codes, 1, 0, opt.nblk)
    master = opt.master.view(opt.nblk, B)
    codes = opt.codes.view(opt.nblk, B)
    step_blocks = 8192
    for a in range(0, opt.nblk, step_blocks):
        b = min(opt.nblk, a + step_blocks)
        mb = master[a:b]
        amax = mb.abs().amax(dim=1)
        # a tensor divisor: torch divides by a Python scalar through its
        # reciprocal, which can be an ulp off the IEEE quotient
        ws = torch.where(amax == 0, torch.ones_like(amax), amax / torch.full_like(amax, 448.0))
        assert torch.equal(opt.scales[a:b].view(torch.int32), ws.view(torch.int32)), a
        wq = (mb / ws[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
        assert torch.equal(codes[a:b], wq), a
    del grads, fp8
    torch.cuda.empty_cache()
