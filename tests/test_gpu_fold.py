"""GPU parity: fold / unfold through the C-ABI against the oracle, bit-exact.

"面向 Blockwise FP8 量化的 ZeRO 优化器设计" §参数布局变换 (fold / unfold),
§块粒度切分 (zero padding to multiples of 128)."""
import numpy as np
import pytest
import torch

import oracle
from blockwise_fp8_zero_fold_gb300 import fp8z1 as F
from tests._gpu import NP_OF, TORCH_OF, bytes_of, lib, to_host  # noqa: F401

pytestmark = pytest.mark.gpu

SHAPE_SETS = {
    "tiny": [(1, 300, 200)],
    "aligned3d": [(3, 256, 384), (2, 128, 1024)],
    "ragged": [(1, 17, 690), (2, 255, 3), (1, 1, 1), (3, 129, 257), (1, 1000, 131)],
    "mixed": [(1, 384, 256), (4, 130, 200), (1, 7, 4096)],
}


def _host_params(shapes, esz, seed):
    rng = np.random.default_rng(seed)
    out = []
    for s in shapes:
        if esz == 4:
            out.append(rng.standard_normal(s).astype(np.float32))
        else:
            out.append(rng.integers(0, 1 << (8 * esz), size=s, dtype=NP_OF[esz]))
    return out


_SIGNED = {4: np.float32, 2: np.int16, 1: np.uint8}  # dtypes torch handles for every size
_SENTINEL = {4: -9.0, 2: 0x3C3C, 1: 0x3C}


def _dev(a):
    return torch.from_numpy(a.view(_SIGNED[a.dtype.itemsize]).copy()).cuda()


@pytest.mark.parametrize("esz", [4, 2, 1])
@pytest.mark.parametrize("name", list(SHAPE_SETS))
def test_fold_unfold_bit_exact(lib, esz, name):
    shapes = SHAPE_SETS[name]
    hp = _host_params(shapes, esz, seed=esz * 7 + len(name))
    L = F.fp8z1_build_layout(shapes, dp_size=3)
    nblk = F.fp8z1_layout_info(L)[0]
    dparams = [_dev(a) for a in hp]
    ptrs = F.param_pointers(dparams)
    ranges = [(0, nblk), (1, nblk), (0, 1), (nblk // 2, nblk), (2, 2)] + [
        F.fp8z1_shard_range(L, r) for r in range(3)]
    for b0, b1 in ranges:
        buf = torch.full(((b1 - b0) * 16384 * esz + 16,), 0x5A, dtype=torch.uint8, device="cuda")
        F.fp8z1_fold(L, ptrs, buf, esz, b0, b1)
        torch.cuda.synchronize()
        want = bytes_of(oracle.fold(shapes, hp, b0, b1))
        got = bytes_of(buf)
        assert np.array_equal(got[:want.size], want), (name, esz, b0, b1)
        assert (got[want.size:] == 0x5A).all()  # nothing written past the shard
        # unfold into sentinel-filled params: only the real elements of [b0, b1)
        outs = [torch.full_like(d, _SENTINEL[esz]) for d in dparams]
        F.fp8z1_unfold(L, buf, F.param_pointers(outs), esz, b0, b1)
        torch.cuda.synchronize()
        ref0 = [np.full(s, _SENTINEL[esz], dtype=_SIGNED[esz]) for s in shapes]
        oracle.unfold(shapes, oracle.fold(shapes, hp, b0, b1).view(_SIGNED[esz]), ref0, b0, b1)
        for o, r0 in zip(outs, ref0):
            assert np.array_equal(bytes_of(o), bytes_of(r0)), (name, esz, b0, b1)
    assert F.fp8z1_device_status(L) == 0


def test_misaligned_param_base_takes_element_path(lib):
    """A param whose base is 4 but not 16-byte aligned (a view at offset 1)."""
    shapes = [(1, 200, 256), (2, 130, 64)]
    hp = _host_params(shapes, 4, seed=5)
    L = F.fp8z1_build_layout(shapes)
    storage = [torch.zeros(int(np.prod(s)) + 1, dtype=torch.float32, device="cuda") for s in shapes]
    views = []
    for st, a, s in zip(storage, hp, shapes):
        v = st[1:].view(s)
        v.copy_(torch.from_numpy(a))
        views.append(v)
    assert all(v.data_ptr() % 16 == 4 for v in views)
    buf = torch.empty(F.fp8z1_layout_info(L)[1], dtype=torch.float32, device="cuda")
    F.fp8z1_fold(L, F.param_pointers(views), buf, 4, 0, F.fp8z1_layout_info(L)[0])
    torch.cuda.synchronize()
    assert np.array_equal(bytes_of(buf), bytes_of(oracle.fold(shapes, hp)))


def test_bad_param_pointer_is_reported_not_touched(lib):
    """A null entry in the pointer array: its blocks are skipped, the status
    word says so, the other params are still folded."""
    shapes = [(1, 128, 128), (1, 256, 128)]
    hp = _host_params(shapes, 4, seed=6)
    L = F.fp8z1_build_layout(shapes)
    d1 = _dev(hp[1])
    ptrs = torch.tensor([0, d1.data_ptr()], dtype=torch.int64, device="cuda")
    buf = torch.full((3 * 16384,), 7.0, dtype=torch.float32, device="cuda")
    F.fp8z1_fold(L, ptrs, buf, 4, 0, 3)
    torch.cuda.synchronize()
    assert F.fp8z1_device_status(L) == F.DEVSTATUS_BADPTR
    assert F.fp8z1_device_status(L) == 0  # read clears
    got = to_host(buf)
    assert (got[:16384] == 7.0).all()
    assert np.array_equal(got[16384:], oracle.fold(shapes, hp, 1, 3))


@pytest.mark.parametrize("esz", [1, 2])
def test_bad_param_pointer_mid_run_unfold(lib, esz):
    """The narrow unfolds copy runs of several blocks per CTA: a null param in
    the middle of a run (blocks 1-2 of 0-4) is skipped and reported, and the
    run carries on with the blocks after it."""
    shapes = [(1, 128, 128), (1, 256, 128), (1, 128, 256)]
    hp = _host_params(shapes, esz, seed=8)
    L = F.fp8z1_build_layout(shapes)
    nblk = F.fp8z1_layout_info(L)[0]
    assert nblk == 5
    buf = _dev(oracle.fold(shapes, hp).view(NP_OF[esz]))
    outs = [torch.full(s, _SENTINEL[esz], dtype=TORCH_OF[esz], device="cuda") for s in shapes]
    ptrs = torch.tensor([outs[0].data_ptr(), 0, outs[2].data_ptr()], dtype=torch.int64, device="cuda")
    F.fp8z1_unfold(L, buf, ptrs, esz, 0, nblk)
    torch.cuda.synchronize()
    assert F.fp8z1_device_status(L) == F.DEVSTATUS_BADPTR
    assert np.array_equal(bytes_of(outs[0]), bytes_of(hp[0]))
    assert np.array_equal(bytes_of(outs[2]), bytes_of(hp[2]))
    assert (bytes_of(outs[1]) == 0x3C).all()  # the sentinel's bytes: untouched


def test_alignment_and_range_errors(lib):
    L = F.fp8z1_build_layout([(1, 300, 200)])
    p = torch.zeros(6 * 16384 + 4, dtype=torch.float32, device="cuda")
    ptrs = F.param_pointers([torch.zeros(300, 200, device="cuda")])
    with pytest.raises(F.Fp8z1Error) as e:
        F.fp8z1_fold(L, ptrs, p.data_ptr() + 4, 4, 0, 6)
    assert e.value.status == F.EALIGN
    with pytest.raises(F.Fp8z1Error) as e:
        F.fp8z1_fold(L, ptrs, p, 4, 0, 7)
    assert e.value.status == F.EINVAL
    with pytest.raises(F.Fp8z1Error) as e:
        F.fp8z1_fold(L, ptrs.data_ptr() + 4, p, 4, 0, 6)
    assert e.value.status == F.EALIGN
