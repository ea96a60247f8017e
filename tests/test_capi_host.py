"""C-ABI host side, no GPU: the library loads, exports every declared symbol,
and its host logic (block LUT, shard ranges, argument checks, loss scaler)
agrees with the oracle."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import oracle
from blockwise_fp8_zero_fold_gb300 import build as fp8build
from blockwise_fp8_zero_fold_gb300 import fp8z1 as F
from blockwise_fp8_zero_fold_gb300 import synth
from tests._golden import parse_shapes, rows

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    fp8build.build()  # nvcc cross-compiles without a GPU
    return F.lib()


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for fn in os.listdir(inc):
        if fn.endswith(".h"):
            text = open(os.path.join(inc, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(fp8z1_\w+)\s*\(", text))
    return names


def test_exports_every_declared_symbol():
    names = _declared()
    assert {"fp8z1_build_layout", "fp8z1_fold", "fp8z1_unfold", "fp8z1_grad_norm",
            "fp8z1_step"} <= names
    lib = C.CDLL(F.lib_path())
    for n in sorted(names):
        assert hasattr(lib, n), n
    assert names <= set(F._SIGS), "binding misses a declared entry point"


def test_checked_env_selects_checked_library():
    """FP8Z1_CHECKED=1 makes the binding load libfp8z1_checked.so (and only
    then); its build flags say so.  No device is needed."""
    import subprocess
    import sys
    fp8build.build(checked=True)
    code = ("from blockwise_fp8_zero_fold_gb300 import fp8z1 as F; "
            "print(F.CHECKED, F.lib_path().endswith('libfp8z1_checked.so'), F.fp8z1_build_flags())")
    for env_value, want in (("1", "True True 1"), ("0", "False False 0")):
        env = dict(os.environ, FP8Z1_CHECKED=env_value)
        r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                           timeout=120)
        assert r.returncode == 0, r.stderr
        assert r.stdout.split()[-3:] == want.split(), r.stdout


def test_checked_build_exports_and_flags():
    """The checked variant exports the same symbols and says it is checked;
    the release build says it is not, reports no misses and refuses the
    table hook (none of this needs a device)."""
    path = fp8build.build(checked=True)
    checked = C.CDLL(path)
    for n in sorted(_declared()):
        assert hasattr(checked, n), n
    checked.fp8z1_build_flags.restype = C.c_int
    assert checked.fp8z1_build_flags() == F.BUILD_CHECKED
    release = C.CDLL(fp8build.lib_path(False))
    release.fp8z1_build_flags.restype = C.c_int
    assert release.fp8z1_build_flags() == 0
    n = C.c_uint64(7)
    assert release.fp8z1_checked_misses(C.byref(n)) == F.OK and n.value == 0
    assert release.fp8z1_checked_misses(None) == F.EINVAL
    L = F.fp8z1_build_layout([(1, 128, 128)], host_only=True)
    e = F.fp8z1_block()
    assert release.fp8z1_checked_set_lut_entry(C.c_void_p(L.handle), C.c_int64(0), C.byref(e)) == F.EINVAL


LUT_CASES = [
    [(1, 300, 200)],
    [(3, 129, 257), (1, 1, 1), (2, 128, 128), (1, 17, 690)],
    synth.workload("moe").shapes,
    synth.ragged_shapes(200, seed=3),
]


@pytest.mark.parametrize("shapes", LUT_CASES, ids=lambda s: str(len(s)))
def test_host_lut_bit_exact_against_oracle(shapes):
    L = F.fp8z1_build_layout(shapes, dp_size=3, host_only=True)
    nblk, padded, real = F.fp8z1_layout_info(L)
    assert nblk == oracle.count_blocks(shapes) and padded == nblk * 16384
    assert real == sum(e * r * c for e, r, c in shapes)
    lut = F.fp8z1_copy_lut(L)
    ref = oracle.build_lut(shapes)
    assert np.array_equal(lut["param"], ref[:, 0])
    assert np.array_equal(lut["expert"], ref[:, 1])
    assert np.array_equal(lut["row_block"], ref[:, 2])
    assert np.array_equal(lut["col_block"], ref[:, 3])
    assert np.array_equal(lut["rows_real"], ref[:, 4])
    assert np.array_equal(lut["cols_real"], ref[:, 5])
    sh = np.array(shapes, dtype=np.int64)
    R, Cc = sh[ref[:, 0], 1], sh[ref[:, 0], 2]
    # element offset of the block's (0,0) element in its row-major param
    assert np.array_equal(lut["src_offset"], (ref[:, 1] * R + 128 * ref[:, 2]) * Cc + 128 * ref[:, 3])
    assert np.array_equal(lut["ld"], Cc)
    for r in range(3):
        assert F.fp8z1_shard_range(L, r) == oracle.shard_range(nblk, 3, r)


@pytest.mark.parametrize("shapes", LUT_CASES, ids=lambda s: str(len(s)))
def test_param_blocks_against_oracle_lut(shapes):
    """fp8z1_param_blocks (where a param's blocks, and so its scales, sit):
    for every param and several ranges, checked against the oracle's block
    table by brute force -- the first block is the first the table gives the
    param, every (e, rb, cb) sits at first + (e*Rb + rb)*Cb + cb, and the
    experts reported held are exactly those whose every block lies in the
    range ("面向 Blockwise FP8 量化的 ZeRO 优化器设计" §总结, §参数布局变换)."""
    from blockwise_fp8_zero_fold_gb300.optimizer import shard_scale_view
    import torch
    ref = oracle.build_lut(shapes)
    nblk = len(ref)
    ranges = [(0, nblk), (0, 0), (nblk, nblk)]
    for dp in (2, 3, 8):
        ranges += [oracle.shard_range(nblk, dp, r) for r in range(dp)]
    rng = np.random.default_rng(len(shapes))
    for _ in range(6):
        a, b = sorted(int(x) for x in rng.integers(0, nblk + 1, 2))
        ranges.append((a, b))
    L = F.fp8z1_build_layout(shapes, host_only=True)
    scales = torch.arange(nblk, dtype=torch.float64)  # scale k holds k
    for p in range(len(shapes)):
        mine = np.flatnonzero(ref[:, 0] == p)
        E = int(ref[mine, 1].max()) + 1
        Rb = int(ref[mine, 2].max()) + 1
        Cb = int(ref[mine, 3].max()) + 1
        for b0, b1 in ranges:
            g = F.fp8z1_param_blocks(L, p, b0, b1)
            assert (g.first_block, g.experts, g.row_blocks, g.col_blocks) == (mine[0], E, Rb, Cb)
            where = g.first_block + (ref[mine, 1] * Rb + ref[mine, 2]) * Cb + ref[mine, 3]
            assert np.array_equal(where, mine)
            held = [e for e in range(E)
                    if all(b0 <= k < b1 for k in mine[ref[mine, 1] == e])]
            want = (held[0], held[-1] + 1) if held else None
            got = (g.e_begin, g.e_end) if g.e_end > g.e_begin else None
            assert got == want, (p, b0, b1)
            v = shard_scale_view(L, scales[b0:b1], b0, b1, p)
            if want is None:
                assert v is None
                continue
            e0, view = v
            assert e0 == want[0] and tuple(view.shape) == (want[1] - want[0], Rb, Cb)
            for k in mine[(ref[mine, 1] >= want[0]) & (ref[mine, 1] < want[1])][:50]:
                e, rb, cb = (int(x) for x in ref[k, 1:4])
                assert view[e - e0, rb, cb].item() == k
    with pytest.raises(F.Fp8z1Error):
        F.fp8z1_param_blocks(L, len(shapes), 0, nblk)
    with pytest.raises(F.Fp8z1Error):
        F.fp8z1_param_blocks(L, 0, 0, nblk + 1)


@pytest.mark.parametrize("row", rows("layout_counts.txt"), ids=lambda r: f"{r[0]}-r{r[4]}")
def test_golden_counts_and_ranges_through_abi(row):
    name, shapes, nblk, dp, rank, b0, b1 = row
    L = F.fp8z1_build_layout(parse_shapes(shapes), dp_size=int(dp), host_only=True)
    assert F.fp8z1_layout_info(L)[0] == int(nblk)
    assert F.fp8z1_shard_range(L, int(rank)) == (int(b0), int(b1))


def test_argument_errors_enqueue_nothing():
    lib = F.lib()
    out = C.c_void_p()
    bad = [[(0, 5, 5)], [(1, -1, 5)], [(1, 5, 1 << 31)]]
    for shapes in bad:
        arr = (F.fp8z1_shape * 1)(F.fp8z1_shape(*shapes[0]))
        assert lib.fp8z1_build_layout(arr, 1, 1, 1, C.byref(out)) == F.EINVAL
        assert out.value is None
    arr = (F.fp8z1_shape * 1)(F.fp8z1_shape(1, 5, 5))
    assert lib.fp8z1_build_layout(arr, 0, 1, 1, C.byref(out)) == F.EINVAL
    assert lib.fp8z1_build_layout(arr, 1, 0, 1, C.byref(out)) == F.EINVAL
    assert lib.fp8z1_build_layout(None, 1, 1, 1, C.byref(out)) == F.EINVAL
    assert lib.fp8z1_build_layout(arr, 1, 1, 0x10, C.byref(out)) == F.EINVAL
    L = F.fp8z1_build_layout([(1, 300, 200)], dp_size=2, host_only=True)
    a, b = C.c_int64(), C.c_int64()
    assert lib.fp8z1_shard_range(L.handle, 2, C.byref(a), C.byref(b)) == F.EINVAL
    assert lib.fp8z1_shard_range(L.handle, -1, C.byref(a), C.byref(b)) == F.EINVAL
    small = np.zeros(2, dtype=F.BLOCK_DTYPE)
    assert lib.fp8z1_copy_lut(L.handle, small.ctypes.data, 2) == F.EINVAL
    # device entry points on a host-only layout: checked and refused before any CUDA call
    buf = np.zeros(64, np.uint8)
    p = buf.ctypes.data
    assert lib.fp8z1_fold(L.handle, p, p, 4, 0, 3, None) == F.ENODEV
    assert lib.fp8z1_fold(L.handle, p, p, 3, 0, 3, None) == F.EINVAL
    assert lib.fp8z1_fold(L.handle, p, p, 4, 2, 1, None) == F.EINVAL
    assert lib.fp8z1_fold(L.handle, p, p, 4, 0, 7, None) == F.EINVAL
    assert lib.fp8z1_unfold(L.handle, p, None, 4, 0, 3, None) == F.EINVAL
    assert lib.fp8z1_grad_norm(L.handle, p, 0, 3, p, p, None) == F.ENODEV
    hp = F.make_hp(1e-3, 0.9, 0.95, 1e-8, 0.1, 1.0, 1024.0, 1)
    assert lib.fp8z1_step(L.handle, C.byref(hp), p, p, p, p, p, p, 0, 3, p, p, None) == F.ENODEV
    for badhp in [F.make_hp(1e-3, 0.9, 0.95, 1e-8, 0.1, 1.0, 1024.0, 0),
                  F.make_hp(1e-3, 1.0, 0.95, 1e-8, 0.1, 1.0, 1024.0, 1),
                  F.make_hp(1e-3, 0.9, 0.95, 0.0, 0.1, 1.0, 1024.0, 1),
                  F.make_hp(1e-3, 0.9, 0.95, 1e-8, 0.1, 1.0, 0.0, 1),
                  F.make_hp(1e-3, 0.9, 0.95, 1e-8, 0.1, 0.0, 1024.0, 1)]:
        assert lib.fp8z1_step(L.handle, C.byref(badhp), p, p, p, p, p, p, 0, 3, p, p, None) == F.EINVAL
    assert lib.fp8z1_norm_reset(None, p, None) == F.EINVAL
    assert lib.fp8z1_norm_reset(p + 4, p, None) == F.EALIGN
    assert lib.fp8z1_norm_reset(p, p + 2, None) == F.EALIGN
    d = np.zeros(16, np.float32).ctypes.data
    assert lib.fp8z1_step_fused_dev(L.handle, None, None, None, p, p, p, p, p, None, p, None, None, 0, 3, p, p,
                                    None) == F.EINVAL
    assert lib.fp8z1_step_fused_dev(L.handle, None, d, None, p, p, p, p, p, None, p, None, None, 0, 3, p, p,
                                    None) == F.ENODEV
    assert lib.fp8z1_device_status(L.handle, C.byref(C.c_uint32())) == F.ENODEV
    assert F.fp8z1_strerror(F.EALIGN) == "misaligned pointer"
    with pytest.raises(F.Fp8z1Error):
        F.fp8z1_shard_range(L, 5)


@pytest.mark.parametrize("row", rows("loss_scale_sequence.txt"))
def test_scaler_matches_oracle_and_golden(row):
    n, s0, flags, scales, steps = row
    s = F.fp8z1_loss_scaler(float(s0), 0, 0, int(n))
    ref = oracle.Scaler(float(s0), int(n))
    got = []
    for f in flags.split(","):
        F.fp8z1_scaler_update(s, int(f))
        ref.update(int(f))
        assert (s.scale, s.step, s.good_steps) == (ref.scale, ref.step, ref.good_steps)
        got.append((s.scale, s.step))
    assert [g[0] for g in got] == [float(x) for x in scales.split(",")]
    assert [g[1] for g in got] == [int(x) for x in steps.split(",")]
    with pytest.raises(F.Fp8z1Error):
        F.fp8z1_scaler_update(F.fp8z1_loss_scaler(0.0, 0, 0, 1), 0)


@pytest.mark.parametrize("dp", [1, 2, 3, 8])
def test_paramwise_split_matches_oracle(dp):
    for shapes in LUT_CASES + [synth.workload("dense").shapes, synth.workload("large").shapes]:
        owner, bucket, padded = F.fp8z1_paramwise_split(shapes, dp)
        o, b = oracle.paramwise_split(shapes, dp)
        assert owner.tolist() == o.tolist() and bucket.tolist() == b.tolist()
        assert padded == dp * int(b.max())


@pytest.mark.parametrize("row", rows("paramwise_split.txt"), ids=lambda r: r[0])
def test_paramwise_split_golden_through_abi(row):
    sizes, dp, owner, buckets, padded = row
    o, b, p = F.fp8z1_paramwise_split([(1, int(x), 1) for x in sizes.split(",")], int(dp))
    assert o.tolist() == [int(x) for x in owner.split(",")]
    assert b.tolist() == [int(x) for x in buckets.split(",")] and p == int(padded)


def test_mx_layout_host():
    shapes = synth.workload("moe").shapes + [(1, 1000, 3008)]
    L = F.fp8z1_mx_build_layout(shapes, dp_size=8, host_only=True)
    groups, elems = F.fp8z1_mx_layout_info(L)
    assert elems == sum(e * r * c for e, r, c in shapes) and groups * 32 == elems
    prev = 0
    for r in range(8):
        g0, g1 = F.fp8z1_mx_shard_range(L, r)
        assert (g0, g1) == oracle.shard_range(groups, 8, r) and g0 == prev
        prev = g1
    assert prev == groups
    with pytest.raises(F.Fp8z1Error):  # C not a multiple of 32
        F.fp8z1_mx_build_layout([(1, 300, 200)], host_only=True)
    lib = F.lib()
    p = np.zeros(8, np.float64).ctypes.data
    hp = F.make_hp(1e-3, 0.9, 0.95, 1e-8, 0.1, 1.0, 1024.0, 1)
    assert lib.fp8z1_mx_step(L.handle, C.byref(hp), p, p, p, p, p, p, 0, 1, p, p, None) == F.ENODEV
    assert lib.fp8z1_mx_grad_norm(L.handle, p, 0, 1, p, p, None) == F.ENODEV
    assert lib.fp8z1_mx_step(L.handle, C.byref(hp), p, p, p, p, p, p, 0, groups + 1, p, p, None) == F.EINVAL


@pytest.mark.parametrize("row", rows("clip_example.txt"))
def test_clip_coef_host_matches_oracle_and_golden(row):
    max_norm, S, grads, sumsq, gnorm, coef, applies, clipped = row
    g, c = F.fp8z1_clip_coef(float(sumsq), float(max_norm), float(S))
    og, oc, oa = oracle.clip_coef(float(sumsq), float(max_norm), float(S))
    assert (g, c) == (og, oc)
    assert g == float(gnorm) and c == pytest.approx(float(coef), rel=1e-15)
    assert (c < 1.0) == bool(int(applies))
    with pytest.raises(F.Fp8z1Error):
        F.fp8z1_clip_coef(-1.0, 1.0, 1.0)


def test_kernel_launch_counter_host():
    """Host-only calls launch nothing; a refused device call launches nothing."""
    n0 = F.fp8z1_kernel_launches()
    L = F.fp8z1_build_layout([(1, 300, 200)], host_only=True)
    F.fp8z1_layout_info(L)
    buf = np.zeros(64, np.uint8)
    assert F.lib().fp8z1_fold(L.handle, buf.ctypes.data, buf.ctypes.data, 4, 0, 1, None) == F.ENODEV
    assert F.fp8z1_kernel_launches() == n0
    assert F.lib().fp8z1_kernel_launches(None) == F.EINVAL


def test_step_scalars_from_hp():
    """The per-step FP32 scalars: each formed in double and rounded once."""
    lr, b1, b2, eps, wd, mx, ls, t = 3e-4, 0.9, 0.95, 1e-8, 0.1, 1.0, 4096.0, 7
    hp = F.make_hp(lr, b1, b2, eps, wd, mx, ls, t)
    sc = F.fp8z1_step_scalars_from_hp(hp)
    f32 = lambda x: float(np.float32(x))  # noqa: E731
    lr, b1, b2, eps, wd = (f32(x) for x in (lr, b1, b2, eps, wd))
    want = dict(beta1=b1, beta2=b2, omb1=f32(1 - b1), omb2=f32(1 - b2), eps=eps,
                step_size=f32(lr / (1 - b1 ** t)), inv_sqrt_bc2=f32(1 / np.sqrt(1 - b2 ** t)),
                decay=f32(1 - lr * wd), max_norm=mx, loss_scale=ls)
    for k, v in want.items():
        assert getattr(sc, k) == v, k
    out = np.zeros(10, np.float32)
    F.fp8z1_step_scalars_from_hp(hp, out)
    assert out[5] == want["step_size"] and out[9] == ls
    with pytest.raises(F.Fp8z1Error) as e:
        F.fp8z1_step_scalars_from_hp(F.make_hp(lr, b1, b2, eps, wd, mx, ls, 0))
    assert e.value.status == F.EINVAL
