"""GPU parity of the widened rows: the quantisation monitors of the fused
step and the MXFP8 variant, against the oracle.

- "FP8训练技术与万亿参数模型优化实践" §1.2: underflow and cosine distortion
  per block (a diagnostic: cosine within 1e-5, underflow counts exact).
- MXFP8 ("面向 Blockwise FP8 量化的 ZeRO 优化器设计" §Blockwise 量化; OCP MX
  v1.0): master / m / v bit-exact (the same FP32 update), E8M0 scales and
  E4M3 codes exact, the norm within 1e-12 of the exact sum."""
import numpy as np
import pytest
import torch

import oracle
from blockwise_fp8_zero_fold_gb300 import fp8z1 as F
from blockwise_fp8_zero_fold_gb300 import synth
from tests._gpu import assert_codes, assert_rel, lib, to_host  # noqa: F401

pytestmark = pytest.mark.gpu
B = 16384


def _hp(**kw):
    d = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=0.5,
             loss_scale=1024.0, step=1)
    d.update(kw)
    return d


@pytest.mark.parametrize("grad_rows", [True, False])
def test_monitors_match_oracle(lib, grad_rows):
    shapes = [(2, 256, 384), (1, 300, 200)]
    rng = np.random.default_rng(5)
    L = F.fp8z1_build_layout(shapes)
    nblk = F.fp8z1_layout_info(L)[0]
    g = [(rng.standard_normal(s) * 1024e-3).astype(np.float32) for s in shapes]
    p = [(rng.standard_normal(s) * 0.02).astype(np.float32) for s in shapes]
    p[0][0, :128, :128] *= 1e-4  # a block with tiny values next to ...
    p[0][0, 0, 0] = 1.0          # ... one large one: many underflow to code 0
    g[0][0, :128, :128] = 0.0    # (no grads there, so the step leaves them tiny)
    dg = [torch.from_numpy(x.copy()).cuda() for x in g]
    dp_ = [torch.from_numpy(x.copy()).cuda() for x in p]
    master = torch.empty(nblk * B, device="cuda")
    F.fp8z1_fold(L, F.param_pointers(dp_), master, 4, 0, nblk)
    mm = torch.zeros(nblk * B, device="cuda")
    vv = torch.zeros(nblk * B, device="cuda")
    q = torch.empty(nblk * B, dtype=torch.uint8, device="cuda")
    sc = torch.empty(nblk, device="cuda")
    cos = torch.full((nblk,), -5.0, device="cuda")
    und = torch.full((nblk,), 12345, dtype=torch.int32, device="cuda")
    s = torch.zeros(1, dtype=torch.float64, device="cuda")
    f = torch.zeros(1, dtype=torch.int32, device="cuda")
    gf = torch.empty(nblk * B, device="cuda")
    F.fp8z1_fold_norm(L, F.param_pointers(dg), gf, 0, nblk, s, f)
    F.fp8z1_step_fused(L, F.make_hp(**_hp()), grad_shard=None if grad_rows else gf,
                       d_grad_params=F.param_pointers(dg) if grad_rows else None, master_shard=master,
                       m_shard=mm, v_shard=vv, fp8_shard=q, scale_shard=sc, block_cos=cos,
                       block_underflow=und, b0=0, b1=nblk, d_sumsq=s, d_found_inf=f)
    torch.cuda.synchronize()
    og, op = oracle.fold(shapes, g), oracle.fold(shapes, p)
    om, ov = np.zeros_like(op), np.zeros_like(op)
    os_, of = oracle.sumsq(og)
    oq, osc, _ = oracle.step(oracle.make_hp(**_hp()), os_, of, og, op, om, ov)
    assert np.array_equal(to_host(q), oq) and np.array_equal(to_host(sc), osc)
    gc, gu = to_host(cos), to_host(und)
    for k in range(nblk):
        c, u = oracle.quant_monitor(op[k * B:(k + 1) * B], oq[k * B:(k + 1) * B], osc[k])
        assert abs(gc[k] - c) <= 1e-5, (k, gc[k], c)
        assert gu[k] == u, (k, gu[k], u)
    # the crafted block: thousands of underflows, yet the one large value keeps
    # its cosine near 1 -- the two monitors see different things
    assert gu[0] > 1000 and (gu[1:] < 10).all()
    assert (gc > 0.995).all()


MX_SHAPES = [(2, 96, 256), (1, 64, 4096), (3, 33, 32)]


def _flat(xs):
    return np.concatenate([x.reshape(-1) for x in xs])


@pytest.mark.parametrize("rank", [0, 1, 2])
def test_mx_step_matches_oracle(lib, rank):
    rng = np.random.default_rng(7 + rank)
    L = F.fp8z1_mx_build_layout(MX_SHAPES, dp_size=3)
    groups, n = F.fp8z1_mx_layout_info(L)
    g0, g1 = F.fp8z1_mx_shard_range(L, rank)
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    p[:32] = 0.0                                  # an all-zero group (scale code 127)
    p[32:64] = (rng.standard_normal(32) * 1e-30).astype(np.float32)  # a tiny group
    p[64:96] = (rng.standard_normal(32) * 1e-40).astype(np.float32)  # subnormal: scale clamps
    m = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    v = np.abs(rng.standard_normal(n) * 1e-8).astype(np.float32)
    m[:96] = 0.0
    v[:96] = 0.0
    sl = slice(g0 * 32, g1 * 32)
    dpp, dm, dv = (torch.from_numpy(x[sl].copy()).cuda() for x in (p, m, v))
    dq = torch.full(((g1 - g0) * 32,), 0xEE, dtype=torch.uint8, device="cuda")
    ds = torch.full((g1 - g0,), 0xEE, dtype=torch.uint8, device="cuda")
    ps, ms, vs = p[sl].copy(), m[sl].copy(), v[sl].copy()
    for t in range(1, 4):
        gh = (rng.standard_normal(n) * 1024e-3).astype(np.float32)
        gh[:96] = 0.0  # the first three groups keep their crafted values
        if t == 2:
            gh[5] = np.inf  # in rank 0's range: every rank skips (the flag is global)
        dg = torch.from_numpy(gh).cuda()
        s = torch.zeros(1, dtype=torch.float64, device="cuda")
        f = torch.zeros(1, dtype=torch.int32, device="cuda")
        for r in range(3):  # every rank's partial, as the all-reduce would
            a, b = F.fp8z1_mx_shard_range(L, r)
            F.fp8z1_mx_grad_norm(L, dg[a * 32:], a, b, s, f)
        hp = _hp(step=t if t < 2 else t - 1)
        F.fp8z1_mx_step(L, F.make_hp(**hp), dg[g0 * 32:], dpp, dm, dv, dq, ds, g0, g1, s, f)
        torch.cuda.synchronize()
        os_, of = oracle.sumsq(gh)
        assert f.item() == of == (1 if t == 2 else 0)
        if not of:
            assert abs(s.item() - os_) <= 1e-12 * os_
        q, sc, skipped = oracle.mx_step(oracle.make_hp(**hp), os_, of, gh[sl].copy(), ps, ms, vs)
        assert skipped == bool(of)
        for a, b, what in [(dpp, ps, "master"), (dm, ms, "m"), (dv, vs, "v")]:
            assert np.array_equal(to_host(a).view(np.uint32), b.view(np.uint32)), what
        if not skipped:
            assert np.array_equal(to_host(dq), q)
            assert np.array_equal(to_host(ds), sc)
    if rank == 0:
        assert to_host(ds)[0] == 127 and (to_host(dq)[:32] == 0).all()
        assert to_host(ds)[2] == 0  # 2^-127: the clamped E8M0 scale


def test_mx_norm_tail_and_errors(lib):
    L = F.fp8z1_mx_build_layout([(1, 1000, 3008)])
    groups, n = F.fp8z1_mx_layout_info(L)
    rng = np.random.default_rng(9)
    g = (rng.standard_normal(n) * 0.1).astype(np.float32)
    dg = torch.from_numpy(g).cuda()
    for g0, g1 in [(0, groups), (3, 700), (5, 6), (groups - 1, groups)]:
        s = torch.zeros(1, dtype=torch.float64, device="cuda")
        f = torch.zeros(1, dtype=torch.int32, device="cuda")
        F.fp8z1_mx_grad_norm(L, dg[g0 * 32:], g0, g1, s, f)
        torch.cuda.synchronize()
        want = oracle.sumsq(g[g0 * 32:g1 * 32])[0]
        assert abs(s.item() - want) <= 1e-12 * want and f.item() == 0
    with pytest.raises(F.Fp8z1Error) as e:
        F.fp8z1_mx_grad_norm(L, dg.data_ptr() + 4, 0, 1, s, f)
    assert e.value.status == F.EALIGN


def test_mx_moe_full_size_sampled(lib):
    """The MoE workload in the MX layout, at full size: two steps, the exact
    global norm, sampled groups against the oracle."""
    w = synth.workload("moe", dp=1)
    L = F.fp8z1_mx_build_layout(w.shapes)
    groups, n = F.fp8z1_mx_layout_info(L)
    dev = torch.device("cuda")

    def flat(kind):
        buf = torch.empty(n, device=dev)
        off = 0
        for t in synth.make_state(w, kind, dev):
            buf[off:off + t.numel()].copy_(t.reshape(-1))
            off += t.numel()
        return buf

    master, mm, vv = flat("master"), flat("m"), flat("v")
    rng = np.random.default_rng(11)
    pick = np.unique(np.concatenate([rng.choice(groups, 400, replace=False), [0, groups - 1]]))
    idx = torch.from_numpy(pick).to(dev)
    state = [to_host(x.view(-1, 32)[idx]).copy() for x in (master, mm, vv)]
    q = torch.empty(n, dtype=torch.uint8, device=dev)
    sc = torch.empty(groups, dtype=torch.uint8, device=dev)
    grad = torch.empty(n, device=dev)
    for t in (1, 2):
        off = 0
        host = []
        for x in synth.make_grads(w, t, dev):
            grad[off:off + x.numel()].copy_(x.reshape(-1))
            off += x.numel()
            host.append(to_host(x))
        s = torch.zeros(1, dtype=torch.float64, device=dev)
        f = torch.zeros(1, dtype=torch.int32, device=dev)
        F.fp8z1_mx_grad_norm(L, grad, 0, groups, s, f)
        hp = _hp(step=t, max_norm=w.max_norm, loss_scale=w.loss_scale)
        F.fp8z1_mx_step(L, F.make_hp(**hp), grad, master, mm, vv, q, sc, 0, groups, s, f)
        torch.cuda.synchronize()
        os_, of = oracle.sumsq_parallel(host, threads=16)
        assert of == 0 and abs(s.item() - os_) <= 1e-12 * os_
        gs = to_host(grad.view(-1, 32)[idx])
        for i in range(len(pick)):
            oq, osc, _ = oracle.mx_step(oracle.make_hp(**hp), os_, 0, gs[i].copy(), state[0][i],
                                        state[1][i], state[2][i])
            assert np.array_equal(to_host(q.view(-1, 32)[int(pick[i])]), oq)
            assert int(sc[int(pick[i])].item()) == int(osc[0])
        for buf, st in zip((master, mm, vv), state):
            assert np.array_equal(to_host(buf.view(-1, 32)[idx]).view(np.uint32), st.view(np.uint32))


# Each MX launch cuts its warp tiles (128 float4 chunks) into one run per CTA:
# runs of 32 tiles on a large buffer, fewer CTAs of smaller runs on a small
# one.  Every element of these buffers is checked, so every run boundary is:
# (3, 1000, 2016) is 11 813 tiles (the last one partial) in 370 runs of ~32;
# (1, 700, 3008) is 4 113 tiles over 304 CTAs of ~13.5; (1, 40, 3008) is 235
# tiles, one per warp.  Rank 1 of 2 starts the shard mid-buffer.
@pytest.mark.parametrize("shape", [(3, 1000, 2016), (1, 700, 3008), (1, 40, 3008)])
@pytest.mark.parametrize("dp,rank", [(1, 0), (2, 1)])
def test_mx_step_every_element(lib, shape, dp, rank):
    rng = np.random.default_rng(shape[1] + 10 * rank)
    L = F.fp8z1_mx_build_layout([shape], dp_size=dp)
    groups, n = F.fp8z1_mx_layout_info(L)
    g0, g1 = F.fp8z1_mx_shard_range(L, rank)
    sl = slice(g0 * 32, g1 * 32)
    ps = (rng.standard_normal(n) * 0.02).astype(np.float32)[sl].copy()
    ms = (rng.standard_normal(n) * 1e-4).astype(np.float32)[sl].copy()
    vs = np.abs(rng.standard_normal(n) * 1e-8).astype(np.float32)[sl].copy()
    dpp, dm, dv = (torch.from_numpy(x.copy()).cuda() for x in (ps, ms, vs))
    dq = torch.full(((g1 - g0) * 32,), 0x7F, dtype=torch.uint8, device="cuda")
    ds = torch.full((g1 - g0,), 0xFF, dtype=torch.uint8, device="cuda")
    for t in (1, 2):
        gh = (rng.standard_normal(n) * 1024e-4).astype(np.float32)
        dg = torch.from_numpy(gh).cuda()
        s = torch.zeros(1, dtype=torch.float64, device="cuda")
        f = torch.zeros(1, dtype=torch.int32, device="cuda")
        F.fp8z1_mx_grad_norm(L, dg, 0, groups, s, f)
        hp = _hp(step=t)
        F.fp8z1_mx_step(L, F.make_hp(**hp), dg[g0 * 32:], dpp, dm, dv, dq, ds, g0, g1, s, f)
        torch.cuda.synchronize()
        os_, of = oracle.sumsq(gh)
        assert of == 0 and abs(s.item() - os_) <= 1e-12 * os_
        q, sc, skipped = oracle.mx_step(oracle.make_hp(**hp), os_, of, gh[sl].copy(), ps, ms, vs)
        assert not skipped
        for a, b, what in [(dpp, ps, "master"), (dm, ms, "m"), (dv, vs, "v")]:
            assert np.array_equal(to_host(a).view(np.uint32), b.view(np.uint32)), what
        assert np.array_equal(to_host(dq), q)
        assert np.array_equal(to_host(ds), sc)


def test_mx_optimizer_steps_and_scaler(lib):
    """MxShardOptimizer over four steps, the third with an inf (skipped: S
    halves, t stays; growth every 2 clean steps), against the oracle's MX
    step and loss scaler ("DeepSpeed ZeRO 优化" §六)."""
    from blockwise_fp8_zero_fold_gb300.optimizer import MxShardOptimizer
    shapes = [(2, 64, 96), (1, 100, 160)]
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=0.5)
    opt = MxShardOptimizer(shapes, loss_scale=1024.0, growth_interval=2, **hp)
    n = sum(e * r * c for e, r, c in shapes)
    assert opt.master.numel() == n
    rng = np.random.default_rng(91)
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    opt.master.copy_(torch.from_numpy(p))
    op, om, ov = p.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    sc = oracle.Scaler(1024.0, 2)
    for t in range(1, 5):
        gh = (rng.standard_normal(n) * sc.scale * 1e-3).astype(np.float32)
        if t == 3:
            gh[n // 2] = np.inf
        found = opt.step(torch.from_numpy(gh).cuda())
        s, fi = oracle.sumsq(gh)
        q, scl, skipped = oracle.mx_step(oracle.make_hp(loss_scale=sc.scale, step=sc.step + 1, **hp), s, fi,
                                         gh, op, om, ov)
        sc.update(int(fi))
        assert found == fi == (1 if t == 3 else 0) and skipped == bool(fi)
        assert (opt.scaler.scale, opt.scaler.step) == (sc.scale, sc.step)
        for a, b in ((opt.master, op), (opt.m, om), (opt.v, ov)):
            assert np.array_equal(to_host(a).view(np.uint32), b.view(np.uint32))
        if not skipped:
            assert np.array_equal(to_host(opt.codes), q) and np.array_equal(to_host(opt.scales), scl)
    assert sc.step == 3 and sc.scale == 1024.0  # x2 after steps 1-2, /2 at the inf


def test_mx_optimizer_resume_is_bit_identical(lib):
    """Checkpoint after two MX steps, reload into a fresh optimizer, carry on:
    state, codes, scales and scaler equal an uninterrupted run."""
    import io

    from blockwise_fp8_zero_fold_gb300.optimizer import MxShardOptimizer
    shapes = [(2, 64, 96), (1, 100, 160)]
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=0.5)
    n = sum(e * r * c for e, r, c in shapes)
    rng = np.random.default_rng(5)
    p = torch.from_numpy((rng.standard_normal(n) * 0.02).astype(np.float32))
    grads = [torch.from_numpy((rng.standard_normal(n) * 1.0).astype(np.float32)).cuda() for _ in range(5)]
    grads[2][n - 5] = float("nan")  # in rank 1's range

    def fresh():
        o = MxShardOptimizer(shapes, dp_size=2, rank=1, loss_scale=1024.0, growth_interval=2, **hp)
        o.master.copy_(o.shard_of(p.cuda()))
        return o

    ref = fresh()
    for g in grads:
        ref.step(ref.shard_of(g))
    first = fresh()
    for g in grads[:2]:
        first.step(first.shard_of(g))
    buf = io.BytesIO()
    torch.save(first.state_dict(), buf)
    buf.seek(0)
    second = MxShardOptimizer(shapes, dp_size=2, rank=1, loss_scale=1.0, growth_interval=2, **hp)
    second.load_state_dict(torch.load(buf))
    for g in grads[2:]:
        second.step(second.shard_of(g))
    for name in ("master", "m", "v", "codes", "scales"):
        assert torch.equal(getattr(ref, name).view(torch.uint8), getattr(second, name).view(torch.uint8)), name
    assert (ref.scaler.scale, ref.scaler.step) == (second.scaler.scale, second.scaler.step)
    st = second.stats()
    assert not st["skipped"] and st["step"] == ref.scaler.step == 4
    assert st["unit_scale_groups"] == int((second.scales == 127).sum())
    with pytest.raises(ValueError):
        MxShardOptimizer(shapes, dp_size=2, rank=0, **hp).load_state_dict(ref.state_dict())


def test_mx_async_steps_equal_synchronous_steps(lib):
    """MxShardOptimizer steps enqueued ahead of their found_inf (t and S
    picked on the device by the previous step's flag) equal the synchronous
    steps over six steps with skips at steps 2 and 3."""
    from blockwise_fp8_zero_fold_gb300.optimizer import MxShardOptimizer
    shapes = [(2, 64, 96), (1, 100, 160)]
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=0.5)
    n = sum(e * r * c for e, r, c in shapes)
    rng = np.random.default_rng(17)
    p = torch.from_numpy((rng.standard_normal(n) * 0.02).astype(np.float32)).cuda()
    gs = [torch.from_numpy((rng.standard_normal(n)).astype(np.float32)).cuda() for _ in range(6)]
    gs[1][11] = float("inf")
    gs[2][n - 3] = float("nan")
    sync = MxShardOptimizer(shapes, loss_scale=1024.0, growth_interval=2, **hp)
    asy = MxShardOptimizer(shapes, loss_scale=1024.0, growth_interval=2, **hp)
    for o in (sync, asy):
        o.master.copy_(p)
    want = [sync.step(g) for g in gs]
    got = []
    for g in gs:
        got += asy.launch_step_async(g)
    got += asy.drain()
    assert want == got == [0, 1, 1, 0, 0, 0]
    assert (asy.scaler.scale, asy.scaler.step) == (sync.scaler.scale, sync.scaler.step)
    for name in ("master", "m", "v", "codes", "scales"):
        assert torch.equal(getattr(sync, name).view(torch.uint8), getattr(asy, name).view(torch.uint8)), name
