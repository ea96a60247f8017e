"""Oracle pins for the widened rows: the param-wise split, the quantisation
monitors and MXFP8.

- "面向 Blockwise FP8 量化的 ZeRO 优化器设计" §参数粒度切分: greedy split of
  whole params over DP buckets, padded to the largest bucket.
- "FP8训练技术与万亿参数模型优化实践" §1.2: underflow and cosine distortion.
- MXFP8 (named in §Blockwise 量化), per the OCP MX specification v1.0."""
import itertools

import numpy as np
import pytest
import torch
from scipy.spatial.distance import cosine as scipy_cosine_distance

import oracle
from tests._golden import rows


@pytest.mark.parametrize("row", rows("paramwise_split.txt"), ids=lambda r: r[0])
def test_paramwise_golden(row):
    sizes, dp, owner, buckets, padded = row
    shapes = [(1, int(x), 1) for x in sizes.split(",")]
    o, b = oracle.paramwise_split(shapes, int(dp))
    assert o.tolist() == [int(x) for x in owner.split(",")]
    assert b.tolist() == [int(x) for x in buckets.split(",")]
    assert int(dp) * b.max() == int(padded)


def test_paramwise_is_a_partition_within_graham_bound_of_the_optimum():
    """Largest-first greedy (LPT): max bucket <= (4/3 - 1/(3D)) * optimum, the
    optimum found by brute force over every assignment."""
    rng = np.random.default_rng(0)
    for _ in range(60):
        dp = int(rng.integers(2, 4))
        n = int(rng.integers(1, 8))
        sizes = [int(x) for x in rng.integers(1, 50, n)]
        shapes = [(1, s, 1) for s in sizes]
        o, b = oracle.paramwise_split(shapes, dp)
        assert all(0 <= x < dp for x in o)
        assert [sum(s for s, w in zip(sizes, o) if w == k) for k in range(dp)] == b.tolist()
        best = min(max(sum(s for s, w in zip(sizes, a) if w == k) for k in range(dp))
                   for a in itertools.product(range(dp), repeat=n))
        assert b.max() >= best
        assert b.max() <= (4 / 3 - 1 / (3 * dp)) * best + 1e-9


def test_monitor_against_scipy_cosine_and_hand_counts():
    rng = np.random.default_rng(1)
    p = (rng.standard_normal(16384) * 0.02).astype(np.float32)
    p[:10] = 1e-9   # far below the smallest code at this scale: they underflow to 0
    p[10] = 0.0     # a true zero is not an underflow
    q, s = oracle.quantise_block(p)
    c, u = oracle.quant_monitor(p, q, s)
    d = oracle.e4m3_decode(q).astype(np.float64) * s
    want = 1.0 - scipy_cosine_distance(p.astype(np.float64), d)
    assert c == pytest.approx(want, abs=1e-12)
    assert 0.995 < c < 1.0
    hand = int(np.sum((p != 0) & (oracle.e4m3_decode(q) == 0)))
    assert u == hand and u >= 10
    # exactly representable values: no distortion, no underflow
    codes = np.arange(0, 0x7F, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes) * np.float32(0.5)
    c, u = oracle.quant_monitor(vals, oracle.e4m3_encode(vals / np.float32(0.5)), 0.5)
    assert c == pytest.approx(1.0, abs=1e-15) and u == 0
    assert oracle.quant_monitor(np.zeros(8, np.float32), np.zeros(8, np.uint8), 1.0) == (1.0, 0)


def test_e8m0_decode_matches_torch():
    codes = torch.arange(0, 255, dtype=torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).float().numpy()
    ours = np.array([oracle.e8m0_decode(int(c)) for c in codes], np.float32)
    assert np.array_equal(ours, ref)
    assert np.isnan(oracle.e8m0_decode(255))


@pytest.mark.parametrize("row", rows("mx_group.txt"), ids=lambda r: r[0])
def test_mx_golden(row):
    v0, v1, v2, sc, c0, c1, c2 = row
    g = np.array([float(v0), float(v1)] + [float(v2)] * 30, np.float32)
    q, s = oracle.mx_quantise(g)
    assert int(s[0]) == int(sc)
    assert [int(q[0]), int(q[1]), int(q[2])] == [int(c0, 16), int(c1, 16), int(c2, 16)]
    assert (q[2:] == q[2]).all()


def test_mx_scale_and_codes_against_definition_and_torch():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(32 * 2000) * np.exp2(rng.integers(-40, 40, 32 * 2000))).astype(np.float32)
    x[:32] = 0.0
    q, s = oracle.mx_quantise(x)
    g = x.reshape(-1, 32).astype(np.float64)
    amax = np.abs(g).max(axis=1)
    for i in range(len(s)):
        X = 2.0 ** (int(s[i]) - 127)
        if amax[i] == 0:
            assert s[i] == 127
            continue
        assert 256 <= amax[i] / X < 512            # X = 2^(floor(log2 amax) - 8)
        y = (g[i] / X).astype(np.float32)
        ref = torch.from_numpy(np.clip(y, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(q[i * 32:(i + 1) * 32], ref)


def test_mx_step_shares_the_update_with_the_block_step():
    rng = np.random.default_rng(3)
    n = 16384
    g = (rng.standard_normal(n) * 1024e-3).astype(np.float32)
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    hp = oracle.make_hp(1e-3, 0.9, 0.95, 1e-8, 0.1, 0.5, 1024.0, 1)
    s, f = oracle.sumsq(g)
    p1, m1, v1 = p.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    p2, m2, v2 = p.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    oracle.step(hp, s, f, g, p1, m1, v1)
    q, sc, skipped = oracle.mx_step(hp, s, f, g, p2, m2, v2)
    assert not skipped
    assert np.array_equal(p1, p2) and np.array_equal(m1, m2) and np.array_equal(v1, v2)
    q2, sc2 = oracle.mx_quantise(p2)
    assert np.array_equal(q, q2) and np.array_equal(sc, sc2)
    g[7] = np.nan
    s, f = oracle.sumsq(g)
    before = p2.copy()
    assert oracle.mx_step(hp, s, f, g, p2, m2, v2)[2] and np.array_equal(before, p2)
