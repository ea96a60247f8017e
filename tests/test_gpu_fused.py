"""GPU parity of the fused forms: fp8z1_fold_norm and fp8z1_step_fused give
the results of the unfused calls ("面向 Blockwise FP8 量化的 ZeRO 优化器设计"
§总结: fold grads -> norm -> update -> quantise -> unfold params), checked
against the oracle and against the unfused entry points."""
import numpy as np
import pytest
import torch

import oracle
from blockwise_fp8_zero_fold_gb300 import fp8z1 as F
from tests._gpu import assert_codes, assert_rel, lib, to_host  # noqa: F401

pytestmark = pytest.mark.gpu
B = 16384

SHAPES = {
    "aligned": [(2, 256, 384), (1, 130, 256)],
    "ragged": [(1, 17, 690), (2, 255, 3), (3, 129, 257), (1, 1000, 131)],
    "mixed": [(1, 300, 200), (2, 128, 1024), (1, 7, 4097)],
}


def _rows(shapes, rng, sigma, dtype=np.float32):
    return [(rng.standard_normal(s) * sigma).astype(dtype) for s in shapes]


def _dev(xs):
    return [torch.from_numpy(x.copy()).cuda() for x in xs]


@pytest.mark.parametrize("name", list(SHAPES))
def test_fold_norm_matches_fold_and_oracle(lib, name):
    shapes = SHAPES[name]
    rng = np.random.default_rng(len(name))
    g = _rows(shapes, rng, 1024e-3)
    dg = _dev(g)
    L = F.fp8z1_build_layout(shapes, dp_size=2)
    nblk = F.fp8z1_layout_info(L)[0]
    ptrs = F.param_pointers(dg)
    for b0, b1 in [(0, nblk), F.fp8z1_shard_range(L, 0), F.fp8z1_shard_range(L, 1), (1, 2), (1, nblk),
                   (0, nblk - 1)]:
        buf = torch.full(((b1 - b0) * B,), 7.0, device="cuda")
        s1 = torch.zeros(1, dtype=torch.float64, device="cuda")
        f1 = torch.zeros(1, dtype=torch.int32, device="cuda")
        F.fp8z1_fold_norm(L, ptrs, buf, b0, b1, s1, f1)
        s2 = torch.zeros(1, dtype=torch.float64, device="cuda")
        f2 = torch.zeros(1, dtype=torch.int32, device="cuda")
        F.fp8z1_fold_norm(L, ptrs, None, b0, b1, s2, f2)
        s3 = torch.zeros(1, dtype=torch.float64, device="cuda")
        f3 = torch.zeros(1, dtype=torch.int32, device="cuda")
        F.fp8z1_grad_norm(L, buf, b0, b1, s3, f3)
        torch.cuda.synchronize()
        want = oracle.fold(shapes, g, b0, b1)
        assert np.array_equal(to_host(buf).view(np.uint32), want.view(np.uint32))
        exact, fe = oracle.sumsq(want)
        assert f1.item() == f2.item() == f3.item() == fe == 0
        # without the store, whole params are summed as flat runs: another order
        assert abs(s1.item() - exact) <= 1e-12 * exact
        assert abs(s2.item() - exact) <= 1e-12 * exact
        assert abs(s3.item() - exact) <= 1e-12 * exact
    assert F.fp8z1_device_status(L) == 0


def test_fold_norm_inf_and_bad_pointer(lib):
    shapes = SHAPES["ragged"]
    rng = np.random.default_rng(3)
    g = _rows(shapes, rng, 1.0)
    g[2][1, 100, 200] = np.nan
    dg = _dev(g)
    L = F.fp8z1_build_layout(shapes)
    nblk = F.fp8z1_layout_info(L)[0]
    s = torch.zeros(1, dtype=torch.float64, device="cuda")
    f = torch.zeros(1, dtype=torch.int32, device="cuda")
    F.fp8z1_fold_norm(L, F.param_pointers(dg), None, 0, nblk, s, f)
    torch.cuda.synchronize()
    assert f.item() == 1 and F.fp8z1_device_status(L) == 0
    # the nan sits in block 7 of param 2: a range that cuts param 2 reads it
    # through the block table, one that holds it whole as flat runs
    p2 = oracle.count_blocks(shapes[:2])
    for b0, b1, want in [(0, p2 + 8, 1), (0, p2 + 7, 0), (p2 + 7, p2 + 8, 1), (1, nblk, 1), (p2 + 8, nblk, 0)]:
        f.zero_()
        F.fp8z1_fold_norm(L, F.param_pointers(dg), None, b0, b1, s, f)
        torch.cuda.synchronize()
        assert f.item() == want, (b0, b1)
    ptrs = F.param_pointers(dg)
    ptrs[1] = 0
    f.zero_()
    F.fp8z1_fold_norm(L, ptrs, None, 0, nblk, s, f)
    torch.cuda.synchronize()
    assert f.item() == 1 and F.fp8z1_device_status(L) == F.DEVSTATUS_BADPTR


def _hp(**kw):
    d = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=0.5,
             loss_scale=1024.0, step=2)
    d.update(kw)
    return F.make_hp(**d)


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("grad_rows,codes_rows,codes_folded",
                         [(True, True, False), (True, True, True), (True, False, True),
                          (False, True, False), (False, True, True), (False, False, True)])
def test_step_fused_equals_step(lib, name, grad_rows, codes_rows, codes_folded):
    shapes = SHAPES[name]
    rng = np.random.default_rng(17)
    L = F.fp8z1_build_layout(shapes, dp_size=2)
    nblk = F.fp8z1_layout_info(L)[0]
    g = _dev(_rows(shapes, rng, 1024e-3))
    p = _dev(_rows(shapes, rng, 0.02))
    m = _dev(_rows(shapes, rng, 1e-4))
    v = [x.abs() for x in _dev(_rows(shapes, rng, 1e-8))]
    gptr = F.param_pointers(g)
    b0, b1 = F.fp8z1_shard_range(L, 1)
    n = (b1 - b0) * B

    def state():
        out = []
        for src in (p, m, v):
            buf = torch.empty(n, device="cuda")
            F.fp8z1_fold(L, F.param_pointers(src), buf, 4, b0, b1)
            out.append(buf)
        return out

    gf = torch.empty(nblk * B, device="cuda")
    s = torch.zeros(1, dtype=torch.float64, device="cuda")
    f = torch.zeros(1, dtype=torch.int32, device="cuda")
    F.fp8z1_fold_norm(L, gptr, gf, 0, nblk, s, f)
    # reference: the unfused step, then unfold
    rp, rm, rv = state()
    rq = torch.empty(n, dtype=torch.uint8, device="cuda")
    rs = torch.empty(b1 - b0, device="cuda")
    F.fp8z1_step(L, _hp(), gf[b0 * B:], rp, rm, rv, rq, rs, b0, b1, s, f)
    r8 = [torch.full(x.shape, 0xEE, dtype=torch.uint8, device="cuda") for x in g]
    F.fp8z1_unfold(L, rq, F.param_pointers(r8), 1, b0, b1)
    # fused
    fp, fm, fv = state()
    fq = torch.full((n,), 0xEE, dtype=torch.uint8, device="cuda") if codes_folded else None
    fs = torch.empty(b1 - b0, device="cuda")
    f8 = [torch.full(x.shape, 0xEE, dtype=torch.uint8, device="cuda") for x in g]
    F.fp8z1_step_fused(L, _hp(), grad_shard=None if grad_rows else gf[b0 * B:],
                       d_grad_params=gptr if grad_rows else None, master_shard=fp, m_shard=fm,
                       v_shard=fv, fp8_shard=fq, d_fp8_params=F.param_pointers(f8) if codes_rows else None,
                       scale_shard=fs, b0=b0, b1=b1, d_sumsq=s, d_found_inf=f)
    torch.cuda.synchronize()
    for a, b in [(rp, fp), (rm, fm), (rv, fv), (rs, fs)]:
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    if codes_folded:
        assert torch.equal(rq, fq)
    if codes_rows:
        for a, b in zip(r8, f8):
            assert torch.equal(a, b)
    assert F.fp8z1_device_status(L) == 0


def test_step_fused_against_oracle_ragged(lib):
    """The fused path end to end (norm from the row-major grads, step reading
    them through the LUT, codes written row-major) against the oracle."""
    shapes = SHAPES["ragged"]
    rng = np.random.default_rng(23)
    L = F.fp8z1_build_layout(shapes)
    nblk = F.fp8z1_layout_info(L)[0]
    gh = _rows(shapes, rng, 65536e-3)
    ph = _rows(shapes, rng, 0.02)
    g, p = _dev(gh), _dev(ph)
    master = torch.empty(nblk * B, device="cuda")
    F.fp8z1_fold(L, F.param_pointers(p), master, 4, 0, nblk)
    mm = torch.zeros(nblk * B, device="cuda")
    vv = torch.zeros(nblk * B, device="cuda")
    sc = torch.empty(nblk, device="cuda")
    f8 = [torch.zeros(x.shape, dtype=torch.uint8, device="cuda") for x in g]
    s = torch.zeros(1, dtype=torch.float64, device="cuda")
    f = torch.zeros(1, dtype=torch.int32, device="cuda")
    F.fp8z1_fold_norm(L, F.param_pointers(g), None, 0, nblk, s, f)
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=0.8,
              loss_scale=65536.0, step=1)
    F.fp8z1_step_fused(L, F.make_hp(**hp), d_grad_params=F.param_pointers(g), master_shard=master,
                       m_shard=mm, v_shard=vv, d_fp8_params=F.param_pointers(f8), scale_shard=sc,
                       b0=0, b1=nblk, d_sumsq=s, d_found_inf=f)
    torch.cuda.synchronize()
    og = oracle.fold(shapes, gh)
    op = oracle.fold(shapes, ph)
    om, ov = np.zeros_like(op), np.zeros_like(op)
    os_, of = oracle.sumsq(og)
    assert abs(s.item() - os_) <= 1e-12 * os_
    q, oscale, _ = oracle.step(oracle.make_hp(**hp), os_, of, og, op, om, ov)
    assert_rel(to_host(master), op, 1e-6, "master")
    assert_rel(to_host(vv), ov, 1e-6, "v")
    assert_rel(to_host(sc), oscale, 1e-6, "scales")
    want = [np.zeros(x.shape, np.uint8) for x in gh]
    oracle.unfold(shapes, q, want)
    for a, b in zip(f8, want):
        assert_codes(to_host(a), b, "row-major codes")
        assert np.array_equal(to_host(a), b)


def test_step_fused_argument_errors(lib):
    L = F.fp8z1_build_layout([(1, 300, 200)])
    t = torch.zeros(6 * B, device="cuda")
    s = torch.zeros(1, dtype=torch.float64, device="cuda")
    f = torch.zeros(1, dtype=torch.int32, device="cuda")
    ptrs = F.param_pointers([torch.zeros(300, 200, device="cuda")])
    common = dict(master_shard=t, m_shard=t, v_shard=t, scale_shard=t, b0=0, b1=6, d_sumsq=s,
                  d_found_inf=f)
    with pytest.raises(F.Fp8z1Error) as e:  # both grad sources
        F.fp8z1_step_fused(L, _hp(), grad_shard=t, d_grad_params=ptrs, fp8_shard=t, **common)
    assert e.value.status == F.EINVAL
    with pytest.raises(F.Fp8z1Error) as e:  # no code destination
        F.fp8z1_step_fused(L, _hp(), d_grad_params=ptrs, **common)
    assert e.value.status == F.EINVAL
    with pytest.raises(F.Fp8z1Error) as e:
        F.fp8z1_step_fused(L, _hp(), d_grad_params=ptrs.data_ptr() + 4, fp8_shard=t, **common)
    assert e.value.status == F.EALIGN


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_fused_path_with_unaligned_param_views(lib, offset):
    """Grads and FP8 weights as views that start 1-3 elements into their
    storage, so every row's misalignment comes from the base address too:
    the fused norm and step read and write them through the unaligned-row
    path and must match the aligned, folded path bit for bit."""
    shapes = [(2, 200, 256), (1, 130, 131), (3, 129, 64)]
    rng = np.random.default_rng(40 + offset)
    L = F.fp8z1_build_layout(shapes)
    nblk = F.fp8z1_layout_info(L)[0]
    gh = _rows(shapes, rng, 1024e-3)
    g_store = [torch.zeros(int(np.prod(s)) + 4, device="cuda") for s in shapes]
    gv = [st[offset:offset + int(np.prod(s))].view(s) for st, s in zip(g_store, shapes)]
    for v, h in zip(gv, gh):
        v.copy_(torch.from_numpy(h))
    c_store = [torch.full((int(np.prod(s)) + 4,), 0xEE, dtype=torch.uint8, device="cuda") for s in shapes]
    cv = [st[offset:offset + int(np.prod(s))].view(s) for st, s in zip(c_store, shapes)]
    p = _dev(_rows(shapes, rng, 0.02))
    ref_g = _dev(gh)  # aligned copies
    s1 = torch.zeros(1, dtype=torch.float64, device="cuda")
    f1 = torch.zeros(1, dtype=torch.int32, device="cuda")
    s2 = torch.zeros(1, dtype=torch.float64, device="cuda")
    f2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    gf = torch.empty(nblk * B, device="cuda")
    F.fp8z1_fold_norm(L, F.param_pointers(ref_g), gf, 0, nblk, s1, f1)
    F.fp8z1_fold_norm(L, F.param_pointers(gv), None, 0, nblk, s2, f2)
    torch.cuda.synchronize()
    assert abs(s1.item() - s2.item()) <= 1e-12 * s1.item() and f1.item() == f2.item() == 0
    s2.copy_(s1)  # one sum for both steps: the update is compared bit for bit

    def state():
        buf = torch.empty(nblk * B, device="cuda")
        F.fp8z1_fold(L, F.param_pointers(p), buf, 4, 0, nblk)
        return buf, torch.zeros(nblk * B, device="cuda"), torch.zeros(nblk * B, device="cuda")

    rp, rm, rv = state()
    rq = torch.empty(nblk * B, dtype=torch.uint8, device="cuda")
    rs = torch.empty(nblk, device="cuda")
    F.fp8z1_step(L, _hp(), gf, rp, rm, rv, rq, rs, 0, nblk, s1, f1)
    r8 = [torch.zeros(s, dtype=torch.uint8, device="cuda") for s in shapes]
    F.fp8z1_unfold(L, rq, F.param_pointers(r8), 1, 0, nblk)
    fp, fm, fv = state()
    fs = torch.empty(nblk, device="cuda")
    F.fp8z1_step_fused(L, _hp(), d_grad_params=F.param_pointers(gv), master_shard=fp, m_shard=fm,
                       v_shard=fv, d_fp8_params=F.param_pointers(cv), scale_shard=fs, b0=0, b1=nblk,
                       d_sumsq=s2, d_found_inf=f2)
    torch.cuda.synchronize()
    for a, b in [(rp, fp), (rm, fm), (rv, fv), (rs, fs)]:
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    for a, b, st, s in zip(r8, cv, c_store, shapes):
        assert torch.equal(a, b)
        n = int(np.prod(s))
        assert (st[:offset] == 0xEE).all() and (st[offset + n:] == 0xEE).all()  # nothing outside the view
    assert F.fp8z1_device_status(L) == 0


@pytest.mark.parametrize("cut", ["whole", "inside_full_run", "across_runs"])
def test_step_mixes_full_and_padded_runs(lib, cut):
    """A layout whose 600-block param of full tiles sits between params with
    padding: the full run goes to the kernel without the padding test, the
    rest to the one that skips the padding-only chunks.  Every form (folded
    and row-major) over whole and cut ranges equals the oracle bit for bit,
    and the padding of master / m / v stays zero."""
    shapes = [(1, 300, 200), (1, 2560, 3840), (2, 129, 257), (1, 256, 256)]
    rng = np.random.default_rng(61)
    L = F.fp8z1_build_layout(shapes)
    nblk = F.fp8z1_layout_info(L)[0]
    b0, b1 = {"whole": (0, nblk), "inside_full_run": (50, 400), "across_runs": (3, nblk - 2)}[cut]
    n = (b1 - b0) * B
    gh = _rows(shapes, rng, 1024e-3)
    ph = _rows(shapes, rng, 0.02)
    mh = _rows(shapes, rng, 1e-4)
    vh = [np.abs(x) for x in _rows(shapes, rng, 1e-8)]
    og, op, om, ov = (oracle.fold(shapes, x, b0, b1) for x in (gh, ph, mh, vh))
    s_exact, fe = oracle.sumsq(og)
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=0.5,
              loss_scale=1024.0, step=3)
    q, oscale, _ = oracle.step(oracle.make_hp(**hp), s_exact, fe, og, op, om, ov)
    want8 = [np.full(x.shape, 0xEE, np.uint8) for x in gh]
    oracle.unfold(shapes, q, want8, b0, b1)
    s = torch.tensor([s_exact], dtype=torch.float64, device="cuda")
    f = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = _dev(gh)
    gf = torch.from_numpy(og).cuda()
    for grad_rows in (False, True):
        p_, m_, v_ = (torch.from_numpy(x).cuda() for x in (oracle.fold(shapes, ph, b0, b1),
                                                            oracle.fold(shapes, mh, b0, b1),
                                                            oracle.fold(shapes, vh, b0, b1)))
        sc = torch.empty(b1 - b0, device="cuda")
        fq = torch.full((n,), 0xEE, dtype=torch.uint8, device="cuda")
        f8 = [torch.full(x.shape, 0xEE, dtype=torch.uint8, device="cuda") for x in gh]
        n0 = F.fp8z1_kernel_launches()
        F.fp8z1_step_fused(L, F.make_hp(**hp), grad_shard=None if grad_rows else gf,
                           d_grad_params=F.param_pointers(g) if grad_rows else None, master_shard=p_,
                           m_shard=m_, v_shard=v_, fp8_shard=fq, d_fp8_params=F.param_pointers(f8),
                           scale_shard=sc, b0=b0, b1=b1, d_sumsq=s, d_found_inf=f)
        # padded blocks before the full run, the run, padded blocks after it
        assert F.fp8z1_kernel_launches() - n0 == {"whole": 3, "inside_full_run": 1, "across_runs": 3}[cut]
        torch.cuda.synchronize()
        for got, want in ((p_, op), (m_, om), (v_, ov), (sc, oscale)):
            assert np.array_equal(to_host(got).view(np.uint32), want.view(np.uint32))
        assert np.array_equal(to_host(fq), q)
        for a, b in zip(f8, want8):
            assert np.array_equal(to_host(a), b)
    assert F.fp8z1_device_status(L) == 0
