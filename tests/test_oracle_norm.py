"""Oracle pins: global grad norm, inf/nan flag and clip coefficient.

"DeepSpeed ZeRO 优化" §七 梯度裁剪 (norm of the loss-scaled grads divided by the
loss scale; clip_coef = max_norm/(norm+1e-6), applied when < 1) and §六 / §九 Q6
(inf or nan in the grads)."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests._golden import rows


def _fsum_squares(g):
    # float32 -> float64 squares are exact (24-bit mantissas), and math.fsum
    # returns the correctly rounded sum: together the exact sum rounded once.
    d = g.astype(np.float64)
    return math.fsum((d * d).tolist())


@pytest.mark.parametrize("case", ["normal", "wide", "subnormal", "huge", "mixed_signs_zeros"])
def test_sumsq_is_exact_sum_rounded_once(case):
    rng = np.random.default_rng(hash(case) % 2**32)
    n = 20000
    if case == "normal":
        g = rng.standard_normal(n).astype(np.float32) * 1e-3
    elif case == "wide":
        g = (rng.standard_normal(n) * np.exp2(rng.integers(-70, 60, n))).astype(np.float32)
    elif case == "subnormal":
        g = (rng.standard_normal(n) * 1e-40).astype(np.float32)
    elif case == "huge":
        g = (rng.standard_normal(n) * 1e30).astype(np.float32)  # squares overflow float32
    else:
        g = rng.standard_normal(n).astype(np.float32)
        g[::3] = 0.0
        g[1::7] = -0.0
    s, f = oracle.sumsq(g)
    assert f == 0
    assert s == _fsum_squares(g)


def test_sumsq_closed_forms():
    assert oracle.sumsq(np.ones(12345, np.float32)) == (12345.0, 0)
    g = np.zeros(1000, np.float32)
    g[417] = np.float32(-3.0000002)
    x = np.float64(np.float32(-3.0000002))
    assert oracle.sumsq(g)[0] == x * x
    assert oracle.sumsq(np.zeros(0, np.float32)) == (0.0, 0)
    # 2^20 copies of 2^-60: exactly 2^-100
    assert oracle.sumsq(np.full(1 << 20, 2.0 ** -60, np.float32))[0] == 2.0 ** -100
    # largest float squared, many times: no overflow in double
    big = np.float32(3.4028235e38)
    assert oracle.sumsq(np.full(1000, big, np.float32))[0] == pytest.approx(1000 * float(big) ** 2, rel=1e-15)


def test_merge_and_parallel_equal_one_shot():
    rng = np.random.default_rng(6)
    parts = [(rng.standard_normal(n) * 10.0 ** rng.integers(-20, 20)).astype(np.float32)
             for n in (1, 1000, 70001, 3)]
    whole = np.concatenate(parts)
    s, f = oracle.sumsq(whole)
    assert oracle.sumsq_parallel(parts, threads=3, chunk=4096) == (s, 0)
    assert s == _fsum_squares(whole)
    parts[2][5] = np.nan
    assert oracle.sumsq_parallel(parts, threads=2, chunk=4096)[1] == 1


def test_chunked_equals_one_shot():
    rng = np.random.default_rng(5)
    g = rng.standard_normal(100003).astype(np.float32)
    acc = oracle.SumsqAccumulator()
    for a, b in [(0, 1), (1, 50000), (50000, 100003)]:
        acc.add(g[a:b])
    assert acc.result() == oracle.sumsq(g)[0]


@pytest.mark.parametrize("bad", [np.inf, -np.inf, np.nan])
def test_found_inf(bad):
    g = np.ones(5000, np.float32)
    g[4321] = bad
    s, f = oracle.sumsq(g)
    assert f == 1
    assert math.isnan(s) if math.isnan(bad) else s == math.inf
    # finite values whose squares overflow float32 are not flagged
    assert oracle.sumsq(np.full(10, 3e38, np.float32))[1] == 0


@pytest.mark.parametrize("row", rows("clip_example.txt"))
def test_clip_golden(row):
    max_norm, S, grads, sumsq, gnorm, coef, applies, clipped = row
    g = np.array([float(x) for x in grads.split(",")], np.float32)
    s, f = oracle.sumsq(g)
    assert s == float(sumsq) and f == 0
    gn, cc, ap = oracle.clip_coef(s, float(max_norm), float(S))
    assert gn == float(gnorm)
    assert cc == pytest.approx(float(coef), rel=1e-15)
    assert ap == bool(int(applies))
    want = np.array([float(x) for x in clipped.split(",")], np.float32)
    got = g / np.float32(S)
    if ap:
        got = got * np.float32(cc)
    assert np.allclose(got, want, rtol=1e-7, atol=0)


@pytest.mark.parametrize("max_norm", [0.05, 1.0, 1e9])
def test_clip_matches_torch_clip_grad_norm(max_norm):
    """torch.nn.utils.clip_grad_norm_ on the unscaled grads (library routine)."""
    rng = np.random.default_rng(9)
    S = 1024.0
    true = [rng.standard_normal(s).astype(np.float32) * 1e-3 for s in [(300, 200), (77,), (5, 5)]]
    stored = [t * np.float32(S) for t in true]
    flat = np.concatenate([s.reshape(-1) for s in stored])
    s, _ = oracle.sumsq(flat)
    gn, cc, ap = oracle.clip_coef(s, max_norm, S)
    params = [torch.nn.Parameter(torch.zeros(t.shape)) for t in true]
    for p, t in zip(params, true):
        p.grad = torch.from_numpy(t.copy())
    total = torch.nn.utils.clip_grad_norm_(params, max_norm, foreach=False)
    assert gn == pytest.approx(float(total), rel=1e-6)
    for p, st in zip(params, stored):
        ours = st / np.float32(S)
        if ap:
            ours = ours * np.float32(cc)
        assert np.allclose(ours, p.grad.numpy(), rtol=2e-6, atol=0)
