"""Oracle pins: the E4M3 codec and per-block quantisation.

E4M3 per the OCP 8-bit floating point specification ("FN": bias 7, no inf,
S.1111.111 NaN, largest finite 448); "FP8训练技术与万亿参数模型优化实践" §1.1
names E4M3; per-block scale from "面向 Blockwise FP8 量化的 ZeRO 优化器设计"
§Blockwise 量化 (one scale per 128x128 block) and §总结 (quantise from the FP32
master); scale = amax/448, or 1 when amax == 0."""
import numpy as np
import pytest
import torch

import oracle
from tests._golden import rows

ALL = np.arange(256, dtype=np.uint8)


def test_decode_matches_torch_float8():
    ours = oracle.e4m3_decode(ALL)
    ref = torch.from_numpy(ALL.copy()).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.isnan(ours[nan]).all()
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _finite_table():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    return codes, oracle.e4m3_decode(codes).astype(np.float64)


def _brute(x):
    """Nearest finite code by exhaustive search; ties -> even code; |x| > 448 -> +-448."""
    codes, vals = _finite_table()
    out = np.empty(x.shape, np.uint8)
    for i, xv in enumerate(x.astype(np.float64)):
        neg = np.signbit(xv)
        a = min(abs(xv), 448.0)
        pos = [(abs(vals[j] - a), j) for j in range(len(codes)) if codes[j] < 0x80]
        best = min(d for d, _ in pos)
        cand = [codes[j] for d, j in pos if d == best]
        c = min(cand) if len(cand) == 1 else [c for c in cand if c % 2 == 0][0]
        out[i] = c | (0x80 if neg else 0)
    return out


def test_encode_brute_force_on_ties_and_neighbours():
    _, vals = _finite_table()
    pos = np.unique(vals[vals >= 0])
    mids = (pos[:-1] + pos[1:]) / 2
    xs = np.concatenate([pos, mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                         np.nextafter(mids.astype(np.float32), np.float32(1e9)),
                         [448.0, 449.0, 463.9, 464.0, 480.0, 1e6, 2.0 ** -10, 2.0 ** -11]])
    xs = xs.astype(np.float32)
    xs = np.concatenate([xs, -xs])
    assert np.array_equal(oracle.e4m3_encode(xs), _brute(xs))


def test_encode_brute_force_random():
    rng = np.random.default_rng(1)
    xs = np.concatenate([rng.uniform(-500, 500, 1500), rng.uniform(-0.02, 0.02, 1500),
                         rng.standard_normal(1000) * 2.0 ** rng.integers(-12, 9, 1000)]).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(xs), _brute(xs))


def test_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(2)
    xs = np.concatenate([rng.uniform(-448, 448, 200000),
                         rng.standard_normal(200000) * 2.0 ** rng.integers(-14, 8, 200000)]).astype(np.float32)
    xs = xs[np.abs(xs) <= 448]
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(xs), ref)


@pytest.mark.parametrize("row", rows("e4m3_codes.txt"), ids=lambda r: r[0])
def test_encode_golden(row):
    x, code = np.float32(float(row[0])), int(row[1], 16)
    assert int(oracle.e4m3_encode(np.array([x]))[0]) == code
    if not (abs(float(x)) > 448):
        assert oracle.lib().oracle_e4m3_encode(float(x)) == code


def _ulp_e4m3(y):
    a = np.abs(y)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    return 2.0 ** (e - 3)


def test_quantise_block_error_bound_and_scale():
    rng = np.random.default_rng(4)
    for sigma in [0.02, 1e-6, 3.0]:
        p = (rng.standard_normal(16384) * sigma).astype(np.float32)
        q, s = oracle.quantise_block(p)
        amax = np.abs(p).max()
        assert s == np.float32(amax) / np.float32(448.0)
        deq = oracle.e4m3_decode(q).astype(np.float64) * s
        y = p.astype(np.float64) / s
        # half an E4M3 step of p/s, times the scale (plus one float32 rounding of p/s)
        bound = 0.5 * _ulp_e4m3(y) * s + np.abs(y) * 2.0 ** -24 * s
        assert (np.abs(p - deq) <= bound * (1 + 1e-12)).all()
        i = int(np.argmax(np.abs(p)))
        assert q[i] in (0x7E, 0xFE)


def test_quantise_zero_block_scale_one():
    q, s = oracle.quantise_block(np.zeros(16384, np.float32))
    assert s == 1.0 and (q == 0).all()
    p = np.zeros(16384, np.float32)
    p[5] = -0.0
    q, s = oracle.quantise_block(p)
    assert s == 1.0 and q[5] == 0x80
