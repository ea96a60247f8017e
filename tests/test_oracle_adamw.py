"""Oracle pins: the fused unscale + clip + AdamW + quantise step.

The pages give no AdamW equations ("面向 Blockwise FP8 量化的 ZeRO 优化器设计"
§ZeRO-1 优化器 names the AdamW moments; §总结 calls the update elementwise);
the reading is standard AdamW with decoupled decay and bias correction.
Pinned against closed forms and against torch.optim.AdamW after
torch.nn.utils.clip_grad_norm_ ("DeepSpeed ZeRO 优化" §三 step order: norm,
unscale+clip, update)."""
import numpy as np
import pytest
import torch

import oracle

B = 16384


def _hp(**kw):
    d = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=1e30,
             loss_scale=1.0, step=1)
    d.update(kw)
    return oracle.make_hp(**d)


def _run(steps, grad_fn, p0, m0=None, v0=None, **kw):
    n = p0.size
    p, m = p0.copy(), (np.zeros(n, np.float32) if m0 is None else m0.copy())
    v = np.zeros(n, np.float32) if v0 is None else v0.copy()
    out = []
    for t in range(1, steps + 1):
        g = grad_fn(t)
        s, f = oracle.sumsq(g)
        codes, scales, skipped = oracle.step(_hp(step=t, **kw), s, f, g, p, m, v)
        out.append((p.copy(), m.copy(), v.copy(), codes, scales, skipped))
    return out


@pytest.mark.parametrize("wd", [0.0, 0.1])
def test_constant_gradient_closed_form(wd):
    """Constant g, no clip, S=1:  m_t = g(1-b1^t), v_t = g^2(1-b2^t),
    mhat = g, sqrt(vhat) = |g|, u = g/(|g|+eps), d = 1 - lr wd,
    p_t = d^t p0 - lr u (1-d^t)/(1-d)   (wd = 0:  p0 - t lr u)."""
    rng = np.random.default_rng(0)
    p0 = (rng.standard_normal(B) * 0.02).astype(np.float32)
    g = (rng.standard_normal(B) * 1e-3).astype(np.float32)
    # the hyper-parameters are FP32 numbers: use exactly those values
    lr, b1, b2, eps, wd32 = (float(np.float32(x)) for x in (1e-3, 0.9, 0.95, 1e-8, wd))
    T = 25
    res = _run(T, lambda t: g, p0, weight_decay=wd)
    g64, p64 = g.astype(np.float64), p0.astype(np.float64)
    u = g64 / (np.abs(g64) + eps)
    d = 1.0 - lr * wd32
    for t in [1, 2, 5, 25]:
        p, m, v = res[t - 1][:3]
        m_cf = g64 * (1 - b1 ** t)
        v_cf = g64 ** 2 * (1 - b2 ** t)
        if wd == 0:
            p_cf = p64 - t * lr * u
        else:
            p_cf = d ** t * p64 - lr * u * (1 - d ** t) / (1 - d)
        assert np.allclose(m, m_cf, rtol=4 * t * 2 ** -23, atol=0)
        assert np.allclose(v, v_cf, rtol=4 * t * 2 ** -23, atol=0)
        # one float32 rounding of p per step, each at most an ulp of the largest
        # |p| along the path, which is below |p0| + t*lr
        assert np.all(np.abs(p - p_cf) <= 3 * t * 2 ** -24 * (np.abs(p64) + t * lr))


def test_zero_gradient_is_pure_decay():
    rng = np.random.default_rng(1)
    p0 = (rng.standard_normal(B) * 0.02).astype(np.float32)
    res = _run(4, lambda t: np.zeros(B, np.float32), p0)
    d = np.float32(1.0 - 1e-3 * 0.1)
    want = p0.copy()
    for t in range(4):
        want = want * d  # m = v = 0 -> update 0, only the decay
        assert np.array_equal(res[t][0], want)
        assert (res[t][1] == 0).all() and (res[t][2] == 0).all()


@pytest.mark.parametrize("max_norm,S", [(1e30, 1.0), (1.0, 1024.0), (0.05, 65536.0)])
def test_matches_torch_adamw_after_clip(max_norm, S):
    """Three steps against torch.optim.AdamW (single-tensor, not fused) fed with
    the unscaled grads clipped by torch.nn.utils.clip_grad_norm_."""
    rng = np.random.default_rng(2)
    n = 2 * B
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    grads = [(rng.standard_normal(n) * 1e-3).astype(np.float32) for _ in range(3)]
    res = _run(3, lambda t: grads[t - 1] * np.float32(S), p0, max_norm=max_norm, loss_scale=S)
    param = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.AdamW([param], lr=1e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1,
                            foreach=False, fused=False)
    for t in range(3):
        param.grad = torch.from_numpy(grads[t].copy())
        torch.nn.utils.clip_grad_norm_([param], max_norm, foreach=False)
        opt.step()
        st = opt.state[param]
        p, m, v = res[t][:3]
        # torch orders the FP32 operations differently (lerp for m, a division by
        # sqrt(bc2)): agreement to a few ulp, far below any dropped term.
        # |p| <= ~0.1 here: 1e-8 is a few ulp; a dropped decay term alone is ~2e-6
        assert np.allclose(p, param.detach().numpy(), rtol=0, atol=1e-8)
        # m and v can cancel: compare at 1e-6 of their scale (a few ulp)
        mr, vr = st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()
        assert np.allclose(m, mr, rtol=0, atol=1e-6 * np.abs(mr).max())
        assert np.allclose(v, vr, rtol=0, atol=1e-6 * np.abs(vr).max())


def test_skip_leaves_state_bit_identical():
    rng = np.random.default_rng(3)
    p = (rng.standard_normal(B) * 0.02).astype(np.float32)
    m = (rng.standard_normal(B) * 1e-4).astype(np.float32)
    v = np.abs(rng.standard_normal(B) * 1e-8).astype(np.float32)
    g = (rng.standard_normal(B) * 1e-3).astype(np.float32)
    g[100] = np.inf
    s, f = oracle.sumsq(g)
    assert f == 1
    p1, m1, v1 = p.copy(), m.copy(), v.copy()
    codes, scales, skipped = oracle.step(_hp(), s, f, g, p1, m1, v1)
    assert skipped
    for a, b in [(p, p1), (m, m1), (v, v1)]:
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_codes_and_scales_come_from_updated_master():
    rng = np.random.default_rng(4)
    n = 3 * B
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    p0[B:2 * B] = 0.0  # a zero block with zero grads stays zero -> scale 1
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    g[B:2 * B] = 0.0
    res = _run(1, lambda t: g, p0)
    p, _, _, codes, scales, _ = res[0]
    for k in range(3):
        q, s = oracle.quantise_block(p[k * B:(k + 1) * B])
        assert scales[k] == s and np.array_equal(codes[k * B:(k + 1) * B], q)
    assert scales[1] == 1.0 and (codes[B:2 * B] == 0).all()
