"""GPU parity of the step with its scalars in device memory
(fp8z1_step_fused_dev) and of the step captured in a CUDA graph
(ShardOptimizer.capture): the same results as the step taking the
hyper-parameters by value, checked against the oracle over several steps
whose t and loss scale change, one of them skipped for an inf
("DeepSpeed ZeRO 优化" §六 / §七; "面向 Blockwise FP8 量化的 ZeRO 优化器设计" §总结)."""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from blockwise_fp8_zero_fold_gb300 import fp8z1 as F
from blockwise_fp8_zero_fold_gb300.optimizer import ShardOptimizer
from tests._gpu import assert_rel, lib, to_host  # noqa: F401

pytestmark = pytest.mark.gpu
B = 16384
SHAPES = [(1, 17, 690), (2, 255, 3), (3, 129, 257), (1, 1000, 131), (2, 256, 384)]
HP = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=0.5)


def _rows(rng, sigma):
    return [(rng.standard_normal(s) * sigma).astype(np.float32) for s in SHAPES]


def _dev(xs):
    return [torch.from_numpy(x.copy()).cuda() for x in xs]


def _as_struct_tensor(sc: F.fp8z1_step_scalars, pinned: bool) -> torch.Tensor:
    t = torch.zeros(C.sizeof(sc) // 4, dtype=torch.float32, pin_memory=pinned)
    C.memmove(t.data_ptr(), C.addressof(sc), C.sizeof(sc))
    return t


@pytest.mark.parametrize("copy", ["host", "none"])
@pytest.mark.parametrize("codes_rows", [True, False])
def test_step_fused_dev_equals_step_fused(lib, copy, codes_rows):
    rng = np.random.default_rng(5)
    L = F.fp8z1_build_layout(SHAPES, dp_size=2)
    b0, b1 = F.fp8z1_shard_range(L, 1)
    n = (b1 - b0) * B
    g = _dev(_rows(rng, 1024e-3))
    p = _dev(_rows(rng, 0.02))
    gptr = F.param_pointers(g)
    s = torch.zeros(1, dtype=torch.float64, device="cuda")
    f = torch.zeros(1, dtype=torch.int32, device="cuda")
    F.fp8z1_fold_norm(L, gptr, None, 0, F.fp8z1_layout_info(L)[0], s, f)
    hp = F.make_hp(loss_scale=1024.0, step=3, **HP)
    outs = []
    for mode in ("value", "dev"):
        master = torch.empty(n, device="cuda")
        F.fp8z1_fold(L, F.param_pointers(p), master, 4, b0, b1)
        mm = torch.full((n,), 1e-4, device="cuda")
        vv = torch.full((n,), 1e-8, device="cuda")
        sc = torch.empty(b1 - b0, device="cuda")
        q = None if codes_rows else torch.empty(n, dtype=torch.uint8, device="cuda")
        f8 = [torch.full(x.shape, 0xEE, dtype=torch.uint8, device="cuda") for x in g] if codes_rows else None
        kw = dict(d_grad_params=gptr, master_shard=master, m_shard=mm, v_shard=vv, fp8_shard=q,
                  d_fp8_params=F.param_pointers(f8) if codes_rows else None, scale_shard=sc, b0=b0, b1=b1,
                  d_sumsq=s, d_found_inf=f)
        if mode == "value":
            F.fp8z1_step_fused(L, hp, **kw)
        else:
            st = F.fp8z1_step_scalars_from_hp(hp)
            if copy == "host":
                h = _as_struct_tensor(st, pinned=True)
                d = torch.zeros_like(h, device="cuda")
                F.fp8z1_step_fused_dev(L, h, d, **kw)
            else:
                d = _as_struct_tensor(st, pinned=False).cuda()
                F.fp8z1_step_fused_dev(L, None, d, **kw)
        torch.cuda.synchronize()
        outs.append([master, mm, vv, sc] + ([q] if q is not None else f8))
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert F.fp8z1_device_status(L) == 0


def test_step_fused_dev_argument_errors(lib):
    L = F.fp8z1_build_layout([(1, 300, 200)])
    t = torch.zeros(6 * B, device="cuda")
    s = torch.zeros(1, dtype=torch.float64, device="cuda")
    f = torch.zeros(1, dtype=torch.int32, device="cuda")
    ptrs = F.param_pointers([torch.zeros(300, 200, device="cuda")])
    d = torch.zeros(10, device="cuda")
    common = dict(d_grad_params=ptrs, master_shard=t, m_shard=t, v_shard=t, fp8_shard=t, scale_shard=t,
                  b0=0, b1=6, d_sumsq=s, d_found_inf=f)
    with pytest.raises(F.Fp8z1Error) as e:
        F.fp8z1_step_fused_dev(L, None, None, **common)
    assert e.value.status == F.EINVAL
    with pytest.raises(F.Fp8z1Error) as e:
        F.fp8z1_step_fused_dev(L, None, d.data_ptr() + 2, **common)
    assert e.value.status == F.EALIGN
    with pytest.raises(F.Fp8z1Error) as e:
        F.fp8z1_step_fused_dev(L, None, d, **dict(common, b1=7))
    assert e.value.status == F.EINVAL


def _oracle_steps(gsteps, ph, loss_scale0, growth):
    """The oracle's run of the same steps: (master, m, v, q, scales) after
    them, and the found_inf of each."""
    op = oracle.fold(SHAPES, ph)
    om, ov = np.zeros_like(op), np.zeros_like(op)
    sc = oracle.Scaler(loss_scale0, growth)
    q = np.zeros(op.size, np.uint8)
    scales = np.ones(op.size // B, np.float32)
    found = []
    for gh in gsteps:
        og = oracle.fold(SHAPES, gh)
        ss, fi = oracle.sumsq(og)
        if not fi:
            hp = oracle.make_hp(loss_scale=sc.scale, step=sc.step + 1,
                                **dict(HP, lr=HP["lr"] / 2 if len(found) == 3 else HP["lr"]))
            q, scales, _ = oracle.step(hp, ss, fi, og, op, om, ov)
        found.append(int(fi))
        sc.update(int(fi))
    return op, om, ov, q, scales, found, sc


@pytest.mark.parametrize("mode", ["patch", "device"])
def test_captured_steps_match_oracle(lib, mode):
    """Four steps through one captured graph, the third with a nan grad (a
    skipped step: S halves, t stays) and the learning rate halved before the
    fourth: master, m, v, scales and the row-major codes match the oracle's
    run of the same steps, and the eager path."""
    rng = np.random.default_rng(11)
    ph = _rows(rng, 0.02)
    scale0, growth = 1024.0, 2
    gsteps = []
    for k in range(4):
        gh = _rows(rng, 1.0)
        gsteps.append(gh)
    gsteps[2][2][1, 100, 30] = np.nan
    # loss-scaled grads as the step sees them: scale g_true by each step's S
    sc = oracle.Scaler(scale0, growth)
    scaled = []
    for gh in gsteps:
        scaled.append([(x * np.float32(sc.scale)).astype(np.float32) for x in gh])
        sc.update(int(any(np.isnan(x).any() for x in gh)))
    op, om, ov, q, oscales, found, osc = _oracle_steps(scaled, ph, scale0, growth)
    assert found == [0, 0, 1, 0]

    from blockwise_fp8_zero_fold_gb300.optimizer import CapturedStep
    if mode == "patch" and not CapturedStep.patch_supported():
        pytest.skip("this torch has no raw CUDA graph handles")
    runs = {}
    for run in ("graph", "eager"):
        opt = ShardOptimizer(SHAPES, loss_scale=scale0, growth_interval=growth, **HP)
        opt.init_state(_dev(ph))
        grads = [torch.zeros(s, device="cuda") for s in SHAPES]
        fp8 = [torch.zeros(s, dtype=torch.uint8, device="cuda") for s in SHAPES]
        cap = opt.capture(grads, fp8, mode=mode) if run == "graph" else None
        if cap is not None:
            assert cap.mode == mode
        got = []
        for k, gh in enumerate(scaled):
            if k == 3:
                opt.hp["lr"] = HP["lr"] / 2  # a schedule step: the graph must follow it
            for t, x in zip(grads, gh):
                t.copy_(torch.from_numpy(x))
            got.append(cap.step() if cap else opt.step(grads, fp8))
        torch.cuda.synchronize()
        assert got == found
        assert (opt.scaler.scale, opt.scaler.step) == (osc.scale, osc.step)
        runs[run] = (opt, fp8)
        assert_rel(to_host(opt.master), op, 1e-6, f"{run} master")
        assert_rel(to_host(opt.m), om, 1e-6, f"{run} m")
        assert_rel(to_host(opt.v), ov, 1e-6, f"{run} v")
        assert_rel(to_host(opt.scales), oscales, 1e-6, f"{run} scales")
        want = [np.zeros(s, np.uint8) for s in SHAPES]
        oracle.unfold(SHAPES, q, want)
        for a, b in zip(fp8, want):
            assert np.array_equal(to_host(a), b)
        assert F.fp8z1_device_status(opt.layout) == 0
    (ga, f8a), (gb, f8b) = runs["graph"], runs["eager"]
    for name in ("master", "m", "v", "scales"):
        assert torch.equal(getattr(ga, name).view(torch.int32), getattr(gb, name).view(torch.int32))
    for a, b in zip(f8a, f8b):
        assert torch.equal(a, b)


def test_patched_graph_with_several_step_launches(lib):
    """A layout whose full-tile run sits between padded params captures three
    step launches (padded, full tiles, padded); fp8z1_graph_step_nodes finds
    all three (and reports the count when the caller's array is short), and
    the patched graph replays two steps equal to the eager path."""
    from blockwise_fp8_zero_fold_gb300.optimizer import CapturedStep
    if not CapturedStep.patch_supported():
        pytest.skip("this torch has no raw CUDA graph handles")
    shapes = [(1, 300, 200), (1, 2560, 3840), (2, 129, 257)]
    rng = np.random.default_rng(29)
    ph = [(rng.standard_normal(s) * 0.02).astype(np.float32) for s in shapes]
    runs = {}
    for run in ("graph", "eager"):
        opt = ShardOptimizer(shapes, loss_scale=1024.0, growth_interval=1000, **HP)
        opt.init_state(_dev(ph))
        grads = [torch.zeros(s, device="cuda") for s in shapes]
        fp8 = [torch.zeros(s, dtype=torch.uint8, device="cuda") for s in shapes]
        cap = opt.capture(grads, fp8, mode="patch") if run == "graph" else None
        if cap is not None:
            assert cap._n_nodes == 3
            n = C.c_int32()
            g = cap.graphs[0].raw_cuda_graph()
            assert F.lib().fp8z1_graph_step_nodes(C.c_void_p(g), None, 0, C.byref(n)) == F.EINVAL and n.value == 3
        r = np.random.default_rng(3)
        for _ in range(2):
            for t, s in zip(grads, shapes):
                t.copy_(torch.from_numpy((r.standard_normal(s) * 1024e-3).astype(np.float32)))
            assert (cap.step() if cap else opt.step(grads, fp8)) == 0
        torch.cuda.synchronize()
        runs[run] = (opt, fp8)
    (a, fa), (b, fb) = runs["graph"], runs["eager"]
    for name in ("master", "m", "v", "scales"):
        assert torch.equal(getattr(a, name).view(torch.int32), getattr(b, name).view(torch.int32)), name
    for x, y in zip(fa, fb):
        assert torch.equal(x, y)
