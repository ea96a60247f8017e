"""Oracle pins: fold / unfold.

Pinned against the view/permute pseudocode of "面向 Blockwise FP8 量化的 ZeRO
优化器设计" §参数布局变换, run with PyTorch CPU ops on zero-padded tensors
(§块粒度切分: pad the quantised dims to multiples of 128), and against the
inverse relation unfold(fold(x)) == x."""
import numpy as np
import pytest
import torch

import oracle

DTYPES = {4: np.float32, 2: np.uint16, 1: np.uint8}


def _rand(shape, esz, rng):
    if esz == 4:
        return rng.standard_normal(shape).astype(np.float32)
    return rng.integers(0, 1 << (8 * esz), size=shape, dtype=DTYPES[esz])


def _pseudocode_fold(x: np.ndarray) -> np.ndarray:
    """The page's fold, applied to x zero-padded up to multiples of 128."""
    E, R, C = x.shape
    Rp, Cp = -(-R // 128) * 128, -(-C // 128) * 128
    t = torch.zeros((E, Rp, Cp), dtype=torch.from_numpy(x).dtype)
    t[:, :R, :C] = torch.from_numpy(x)
    w = (t.view(t.shape[0], t.shape[1] // 128, 128, t.shape[2] // 128, 128)
         .permute(0, 1, 3, 2, 4).contiguous().view(-1, 128, 128))
    return w.numpy().reshape(-1)


def _pseudocode_unfold(buf: np.ndarray, E, R, C) -> np.ndarray:
    Rp, Cp = -(-R // 128) * 128, -(-C // 128) * 128
    w = torch.from_numpy(buf.copy())
    t = (w.view(E, Rp // 128, Cp // 128, 128, 128).permute(0, 1, 3, 2, 4)
         .contiguous().view(E, Rp, Cp))
    return t[:, :R, :C].numpy()


SHAPE_SETS = [
    [(1, 300, 200)],
    [(3, 129, 257)],
    [(1, 1, 1), (2, 128, 128), (1, 17, 690), (2, 255, 3)],
    [(1, 384, 256), (1, 1000, 131)],
]


@pytest.mark.parametrize("esz", [4, 2, 1])
@pytest.mark.parametrize("shapes", SHAPE_SETS, ids=lambda s: str(len(s)))
def test_fold_matches_pseudocode(esz, shapes):
    rng = np.random.default_rng(len(shapes) * 10 + esz)
    xs = [_rand(s, esz, rng) for s in shapes]
    want = np.concatenate([_pseudocode_fold(x) for x in xs])
    got = oracle.fold(shapes, xs)
    assert got.dtype == xs[0].dtype
    assert np.array_equal(got.view(np.uint8), want.view(np.uint8))


@pytest.mark.parametrize("esz", [4, 2, 1])
@pytest.mark.parametrize("shapes", SHAPE_SETS, ids=lambda s: str(len(s)))
def test_unfold_inverts_fold_and_matches_pseudocode(esz, shapes):
    rng = np.random.default_rng(100 + len(shapes) * 10 + esz)
    xs = [_rand(s, esz, rng) for s in shapes]
    buf = oracle.fold(shapes, xs)
    sentinel = {4: np.float32(-7.0), 2: np.uint16(0xBEEF), 1: np.uint8(0xA5)}[esz]
    outs = [np.full(s, sentinel, dtype=xs[0].dtype) for s in shapes]
    oracle.unfold(shapes, buf, outs)
    off = 0
    for x, o, (E, R, C) in zip(xs, outs, shapes):
        assert np.array_equal(o.view(np.uint8), x.view(np.uint8))
        nb = E * (-(-R // 128)) * (-(-C // 128))
        ref = _pseudocode_unfold(buf[off * 16384:(off + nb) * 16384], E, R, C)
        assert np.array_equal(ref.view(np.uint8), x.view(np.uint8))
        off += nb


def test_fold_subrange_is_slice_and_padding_is_zero():
    shapes = [(2, 200, 300), (1, 130, 5)]
    rng = np.random.default_rng(7)
    xs = [_rand(s, 4, rng) + 10.0 for s in shapes]  # no real element is zero
    full = oracle.fold(shapes, xs)
    nblk = oracle.count_blocks(shapes)
    for b0, b1 in [(0, nblk), (1, 4), (5, nblk), (3, 3)]:
        part = oracle.fold(shapes, xs, b0, b1)
        assert np.array_equal(part, full[b0 * 16384:b1 * 16384])
    lut = oracle.build_lut(shapes)
    blocks = full.reshape(nblk, 128, 128)
    for k, (p, e, rb, cb, rr, cr) in enumerate(lut):
        assert (blocks[k, rr:, :] == 0).all() and (blocks[k, :, cr:] == 0).all()
        assert (blocks[k, :rr, :cr] != 0).all()


def test_unfold_subrange_writes_only_its_blocks():
    shapes = [(1, 300, 200)]
    rng = np.random.default_rng(3)
    x = _rand(shapes[0], 1, rng)
    buf = oracle.fold(shapes, [x])
    out = np.full(shapes[0], 0xEE, dtype=np.uint8)
    oracle.unfold(shapes, buf[2 * 16384:4 * 16384], [out], 2, 4)  # blocks (rb=1, cb=0..1)
    assert np.array_equal(out[0, 128:256, :], x[0, 128:256, :])
    assert (out[0, :128, :] == 0xEE).all() and (out[0, 256:, :] == 0xEE).all()


def test_brute_force_many_small_shapes():
    rng = np.random.default_rng(11)
    for _ in range(12):
        shapes = [(int(rng.integers(1, 4)), int(rng.integers(1, 301)), int(rng.integers(1, 301)))
                  for _ in range(int(rng.integers(1, 4)))]
        xs = [_rand(s, 2, rng) for s in shapes]
        want = np.concatenate([_pseudocode_fold(x) for x in xs])
        assert np.array_equal(oracle.fold(shapes, xs), want)
