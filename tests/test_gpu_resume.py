"""Checkpoint / resume: k steps, save, reload into a fresh optimizer, carry
on -- bit-identical to an uninterrupted run.  The state is the four 1-D block
buffers plus t and S; the norm reduction is deterministic, so resuming
reproduces every bit."""
import io
import json

import numpy as np
import pytest
import torch

from blockwise_fp8_zero_fold_gb300 import fp8z1 as F
from blockwise_fp8_zero_fold_gb300 import synth
from blockwise_fp8_zero_fold_gb300.optimizer import ShardOptimizer
from tests._gpu import lib  # noqa: F401

pytestmark = pytest.mark.gpu


def _make(w, rank):
    opt = ShardOptimizer(w.shapes, dp_size=w.dp, rank=rank, loss_scale=w.loss_scale,
                         growth_interval=2, **{k: v for k, v in w.hp().items() if k != "loss_scale"})
    return opt


def test_resume_is_bit_identical(lib):
    w = synth.workload("tiny", shapes=[(2, 300, 520), (1, 1000, 131)], dp=2, rank=1,
                       m_sigma=1e-4, v_sigma=1e-8, max_norm=0.3)
    fp8 = [torch.zeros(s, dtype=torch.uint8, device="cuda") for s in w.shapes]

    def run(opt, steps):
        for t in steps:
            g = synth.make_grads(w, t, "cuda")
            if t == 3:
                g[1][0, 5, 7] = float("nan")  # a skipped step inside the run (param 1 is in rank 1's range)
            opt.step(g, fp8)

    ref = _make(w, 1)
    ref.init_state(*(synth.make_state(w, k, "cuda") for k in ("master", "m", "v")))
    run(ref, range(1, 6))

    first = _make(w, 1)
    first.init_state(*(synth.make_state(w, k, "cuda") for k in ("master", "m", "v")))
    run(first, range(1, 3))
    buf = io.BytesIO()
    torch.save(first.state_dict(), buf)
    del first
    buf.seek(0)
    second = _make(w, 1)
    second.load_state_dict(torch.load(buf))
    run(second, range(3, 6))
    torch.cuda.synchronize()
    for name in ("master", "m", "v", "codes", "scales"):
        a, b = getattr(ref, name), getattr(second, name)
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), name
    assert (ref.scaler.scale, ref.scaler.step, ref.scaler.good_steps) == \
        (second.scaler.scale, second.scaler.step, second.scaler.good_steps)
    assert ref.scaler.step == 4  # one of the five steps was skipped
    with pytest.raises(ValueError):
        _make(synth.workload("tiny"), 0).load_state_dict(ref.state_dict())


@pytest.mark.parametrize("max_norm", [1e30, 0.05])
def test_step_from_host_matches_device_path(lib, max_norm):
    """Grads from pinned host memory and FP8 weights back to it, with the
    copies overlapped: the same state as the device-resident step.  With
    clipping off the result is bit-identical; with clipping on the chunked
    norm adds its partials in another order, so 1e-6 relative."""
    w = synth.workload("tiny", shapes=[(3, 512, 384), (1, 1000, 131)], dp=1, rank=0,
                       m_sigma=1e-4, v_sigma=1e-8, max_norm=max_norm)
    ref = _make(w, 0)
    host = _make(w, 0)
    for o in (ref, host):
        o.init_state(*(synth.make_state(w, k, "cuda") for k in ("master", "m", "v")))
    fp8 = [torch.zeros(s, dtype=torch.uint8, device="cuda") for s in w.shapes]
    hfp8 = [torch.zeros(s, dtype=torch.uint8, pin_memory=True) for s in w.shapes]
    hsc = torch.zeros(host.nblk, dtype=torch.float32, pin_memory=True)
    for t in (1, 2):
        g = synth.make_grads(w, t, "cuda")
        hg = [x.cpu().pin_memory() for x in g]
        assert ref.step(g, fp8) == 0
        assert host.step_from_host(hg, hfp8, hsc, target_blocks=7) == 0
    torch.cuda.synchronize()
    for name in ("master", "m", "v", "scales"):
        a, b = getattr(ref, name), getattr(host, name)
        if max_norm > 1e20:
            assert torch.equal(a.view(torch.int32), b.view(torch.int32)), name
        else:
            assert torch.allclose(a, b, rtol=1e-6, atol=0), name
    if max_norm > 1e20:
        for a, b in zip(fp8, hfp8):
            assert torch.equal(a.cpu(), b)
        assert torch.equal(hsc, ref.scales.cpu())
    assert host.scaler.step == 2
    with pytest.raises(ValueError):
        _make(synth.workload("tiny"), 0).step_from_host([], [])


def test_pipelined_steps_from_host(lib):
    """Four steps from host buffers enqueued back to back (wait=False: step
    k+1's grads go in while step k's update and copies back run), the third
    skipped for a nan: the same state, FP8 weights, scales and loss scaler
    as the device-resident path stepping one at a time."""
    w = synth.workload("tiny", shapes=[(3, 512, 384), (1, 1000, 131), (2, 130, 260)], dp=1, rank=0,
                       m_sigma=1e-4, v_sigma=1e-8, max_norm=1e30)
    ref, host = _make(w, 0), _make(w, 0)
    for o in (ref, host):
        o.init_state(*(synth.make_state(w, k, "cuda") for k in ("master", "m", "v")))
    fp8 = [torch.zeros(s, dtype=torch.uint8, device="cuda") for s in w.shapes]
    hfp8 = [torch.zeros(s, dtype=torch.uint8, pin_memory=True) for s in w.shapes]
    hsc = torch.zeros(host.nblk, dtype=torch.float32, pin_memory=True)
    hgs, found = [], []
    for t in range(1, 5):
        g = synth.make_grads(w, t, "cuda")
        if t == 3:
            g[2][1, 7, 9] = float("nan")
        hgs.append([x.cpu().pin_memory() for x in g])
        found.append(ref.step(g, fp8))
    for hg in hgs:
        assert host.step_from_host(hg, hfp8, hsc, target_blocks=3, wait=False) is None
    assert host.finish_host_step() == 0 and host.finish_host_step() is None
    assert found == [0, 0, 1, 0]
    assert (host.scaler.scale, host.scaler.step) == (ref.scaler.scale, ref.scaler.step) and ref.scaler.step == 3
    for name in ("master", "m", "v", "scales"):
        assert torch.equal(getattr(ref, name).view(torch.int32), getattr(host, name).view(torch.int32)), name
    for a, b in zip(fp8, hfp8):
        assert torch.equal(a.cpu(), b)
    assert torch.equal(hsc, ref.scales.cpu())
    with pytest.raises(RuntimeError):  # no device-path step while a host step is in flight
        host.step_from_host(hgs[0], hfp8, hsc, target_blocks=3, wait=False)
        host.step(synth.make_grads(w, 5, "cuda"), fp8)
    host.finish_host_step()


def test_stats_report_the_step(lib):
    import oracle
    w = synth.workload("tiny", dp=1, rank=0, max_norm=0.05)
    opt = _make(w, 0)
    opt.init_state(synth.make_state(w, "master", "cuda"))
    g = synth.make_grads(w, 1, "cuda")
    assert opt.step(g) == 0
    st = opt.stats(loss_scale=w.loss_scale)
    s, _ = oracle.sumsq(np.concatenate([x.cpu().numpy().ravel() for x in g]))
    gn, cc, ap = oracle.clip_coef(s, w.max_norm, w.loss_scale)
    assert st["global_norm"] == pytest.approx(gn, rel=1e-12)
    assert st["clip_coef"] == pytest.approx(cc, rel=1e-12)
    assert st["clipped"] == ap and not st["skipped"] and st["step"] == 1
    assert st["unit_scale_blocks"] == int((opt.scales == 1.0).sum())
    buf = io.StringIO()
    line = opt.log_step(buf, step_ms=0.5, note="x")
    assert json.loads(buf.getvalue()) == line and line["note"] == "x"
    assert line["elem_per_s"] == pytest.approx(opt.nblk * 16384 / 0.5e-3)


def test_unit_scale_blocks_counts_zero_blocks(lib):
    """A block whose masters, moments and grads are all zero stays zero and
    takes scale 1 (the scale when amax = 0); stats() counts such blocks."""
    w = synth.workload("tiny", shapes=[(4, 128, 128)], dp=1, rank=0, max_norm=1e30)
    opt = _make(w, 0)
    master = synth.make_state(w, "master", "cuda")
    master[0][1].zero_()
    master[0][3].zero_()
    opt.init_state(master)
    g = synth.make_grads(w, 1, "cuda")
    g[0][1].zero_()
    g[0][3].zero_()
    assert opt.step(g) == 0
    assert opt.stats()["unit_scale_blocks"] == 2


# padded runs only (36 full tiles are too few for a full-tile run); and a
# 512-block full-tile param between padded ones, so that each step is a
# full-tile launch and padded launches, each picking its scalars by the flag
ASYNC_SHAPES = {"padded": [(3, 512, 384), (1, 1000, 131), (2, 130, 260)],
                "full_and_padded": [(1, 1000, 131), (1, 4096, 2048), (2, 130, 260)]}


@pytest.mark.parametrize("layout_kind", list(ASYNC_SHAPES))
def test_async_steps_equal_synchronous_steps(lib, layout_kind):
    """Eight steps enqueued ahead of their found_inf (launch_step_async: each
    step's t and S picked on the device by the previous step's flag), with
    skips at steps 3, 4 and 7 and the scale growing every 2 clean steps: the
    state, FP8 weights, scales and loss scaler equal the synchronous path's."""
    w = synth.workload("tiny", shapes=ASYNC_SHAPES[layout_kind], dp=1, rank=0,
                       m_sigma=1e-4, v_sigma=1e-8, max_norm=0.5)
    sync, asy = _make(w, 0), _make(w, 0)
    for o in (sync, asy):
        o.init_state(*(synth.make_state(w, k, "cuda") for k in ("master", "m", "v")))
    f_sync = [torch.zeros(s, dtype=torch.uint8, device="cuda") for s in w.shapes]
    f_asy = [torch.zeros(s, dtype=torch.uint8, device="cuda") for s in w.shapes]
    bad = {3, 4, 7}
    gs = []
    for t in range(1, 9):
        g = synth.make_grads(w, t, "cuda")
        if t in bad:
            g[t % 3][0, 3, 5] = float("nan")
        gs.append(g)
    want = [sync.step(g, f_sync) for g in gs]
    got = []
    g_dev = [torch.empty_like(x) for x in gs[0]]
    g_ptrs, f_ptrs = asy.pointers(g_dev), asy.pointers(f_asy)  # the loop passes pointer arrays
    for g in gs:
        for d, x in zip(g_dev, g):
            d.copy_(x)  # the same grad tensors every step, refilled in stream order
        got += asy.launch_step_async(g_ptrs, f_ptrs)
    got += asy.drain()
    assert want == got == [int(t in bad) for t in range(1, 9)]
    assert (asy.scaler.scale, asy.scaler.step, asy.scaler.good_steps) == \
        (sync.scaler.scale, sync.scaler.step, sync.scaler.good_steps)
    for name in ("master", "m", "v", "scales"):
        assert torch.equal(getattr(sync, name).view(torch.int32), getattr(asy, name).view(torch.int32)), name
    for a, b in zip(f_sync, f_asy):
        assert torch.equal(a, b)
    assert asy.stats()["step"] == 5 and F.fp8z1_device_status(asy.layout) == 0
    with pytest.raises(RuntimeError):  # no synchronous step while async steps are in flight
        asy.launch_step_async(g_dev, f_asy)
        asy.step(g_dev, f_asy)
    asy.drain()


@pytest.mark.parametrize("mode", ["sync", "async"])
def test_two_ranks_through_the_norm_hook(lib, mode):
    """Ranks 0 and 1 of DP = 2 on one GPU: each rank's norm hook adds the
    other rank's partial sum of squares and ORs its flag, as the all-reduce
    of "DeepSpeed ZeRO 优化" §七 would, and both write their blocks' codes
    into the same FP8 weights (the all-gather).  With a nan in rank 1's
    range on step 2, both ranks skip it.  Their shards and the FP8 weights
    equal one whole-buffer optimizer's, bit for bit (clipping off: the update
    does not depend on how the sum was grouped)."""
    base = dict(shapes=[(3, 512, 384), (1, 1000, 131)], m_sigma=1e-4, v_sigma=1e-8, max_norm=1e30)
    w1 = synth.workload("tiny", dp=1, rank=0, **base)
    w2 = synth.workload("tiny", dp=2, rank=0, **base)
    ref = _make(w1, 0)
    ranks = [_make(w2, r) for r in (0, 1)]
    for o in [ref] + ranks:
        o.init_state(*(synth.make_state(w1, k, "cuda") for k in ("master", "m", "v")))
    assert ranks[1].b0 <= oracle_block_of_param(w2, 1) < ranks[1].b1
    fp8_ref = [torch.zeros(s, dtype=torch.uint8, device="cuda") for s in w1.shapes]
    fp8 = [torch.zeros(s, dtype=torch.uint8, device="cuda") for s in w1.shapes]
    part = torch.zeros(2, dtype=torch.float64, device="cuda")
    pflag = torch.zeros(2, dtype=torch.int32, device="cuda")

    def hook_for(r):
        def hook(s, f):  # add the other rank's partial, OR its flag
            s.add_(part[1 - r:2 - r])
            torch.maximum(f, pflag[1 - r:2 - r], out=f)
        return hook

    for r, o in enumerate(ranks):
        o.norm_hook = hook_for(r)
    got = [[], []]
    for t in range(1, 4):
        g = synth.make_grads(w1, t, "cuda")
        if t == 2:
            g[1][0, 5, 7] = float("nan")
        ref.step(g, fp8_ref)
        part.zero_()
        pflag.zero_()
        for r, o in enumerate(ranks):  # each rank's own partial, as it would send it
            F.fp8z1_fold_norm(o.layout, F.param_pointers(g), None, o.b0, o.b1, part[r:r + 1], pflag[r:r + 1])
        for r, o in enumerate(ranks):
            if mode == "sync":
                got[r].append(o.step(g, fp8))
            else:
                got[r] += o.launch_step_async(g, fp8)
    if mode == "async":
        for r, o in enumerate(ranks):
            got[r] += o.drain()
    torch.cuda.synchronize()
    assert got[0] == got[1] == [0, 1, 0]
    for o in ranks:
        assert (o.scaler.scale, o.scaler.step) == (ref.scaler.scale, ref.scaler.step) and o.scaler.step == 2
        sl = slice(o.b0 * 16384, o.b1 * 16384)
        for name in ("master", "m", "v"):
            assert torch.equal(getattr(o, name).view(torch.int32), getattr(ref, name)[sl].view(torch.int32)), name
        assert torch.equal(o.scales, ref.scales[o.b0:o.b1])
    for a, b in zip(fp8, fp8_ref):
        assert torch.equal(a, b)


def oracle_block_of_param(w, p):
    """The first block of param p in the workload's block order."""
    import oracle
    return oracle.count_blocks(w.shapes[:p])
