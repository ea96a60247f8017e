"""The pins catch planted mistakes.

Each case below copies the oracle's C source, plants one plausible mistake
(a dropped term, a wrong sign, a swapped loop, a wrong constant, a rounding
or saturation slip), builds it, and runs a battery of independent pins
against it -- PyTorch's view/permute fold, math.fsum, torch.optim.AdamW with
clip_grad_norm_, torch.float8_e4m3fn / float8_e8m0fnu, scipy's cosine, the
hand-derived golden files.  Every mistake must fail at least one pin, and the
unmodified oracle must pass them all.  The mistakes are planted on the CPU
only, and each keeps every memory access in bounds."""
import math
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch
from scipy.spatial.distance import cosine as scipy_cosine_distance

import oracle
from tests._golden import parse_shapes, rows

SRC = os.path.join(os.path.dirname(oracle.__file__), "fp8z1_oracle.c")


# ---------------------------------------------------------------------------
# the pin battery (independent of the oracle's own arithmetic)

def _pad_fold(x):
    E, R, Cc = x.shape
    t = torch.zeros((E, -(-R // 128) * 128, -(-Cc // 128) * 128), dtype=torch.from_numpy(x).dtype)
    t[:, :R, :Cc] = torch.from_numpy(x)
    return (t.view(E, t.shape[1] // 128, 128, t.shape[2] // 128, 128).permute(0, 1, 3, 2, 4)
            .contiguous().view(-1).numpy())


def pin_fold():
    rng = np.random.default_rng(0)
    shapes = [(2, 200, 300), (1, 17, 129)]
    xs = [rng.standard_normal(s).astype(np.float32) + 5 for s in shapes]
    want = np.concatenate([_pad_fold(x) for x in xs])
    got = oracle.fold(shapes, xs)
    if not np.array_equal(got, want):
        return False
    outs = [np.zeros(s, np.float32) for s in shapes]
    oracle.unfold(shapes, got, outs)
    return all(np.array_equal(a, b) for a, b in zip(outs, xs))


def pin_layout():
    for name, shapes, nblk, dp, rank, b0, b1 in rows("layout_counts.txt"):
        sh = parse_shapes(shapes)
        if oracle.count_blocks(sh) != int(nblk):
            return False
        if oracle.shard_range(int(nblk), int(dp), int(rank)) != (int(b0), int(b1)):
            return False
    return True


def pin_sumsq():
    rng = np.random.default_rng(1)
    g = (rng.standard_normal(5001) * 3).astype(np.float32)
    d = g.astype(np.float64)
    return oracle.sumsq(g) == (math.fsum((d * d).tolist()), 0) and oracle.sumsq(
        np.array([1.0, np.inf], np.float32))[1] == 1


def pin_clip_and_adamw():
    rng = np.random.default_rng(2)
    n = 2 * 16384
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    S = 1024.0
    ok = True
    for max_norm in (1e30, 0.05):
        p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
        param = torch.nn.Parameter(torch.from_numpy(p0.copy()))
        opt = torch.optim.AdamW([param], lr=1e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1,
                                foreach=False, fused=False)
        for t in range(1, 4):
            g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
            gs = g * np.float32(S)
            s, f = oracle.sumsq(gs)
            oracle.step(oracle.make_hp(1e-3, 0.9, 0.95, 1e-8, 0.1, max_norm, S, t), s, f, gs, p, m, v)
            param.grad = torch.from_numpy(g.copy())
            torch.nn.utils.clip_grad_norm_([param], max_norm, foreach=False)
            opt.step()
            ok &= bool(np.allclose(p, param.detach().numpy(), rtol=0, atol=1e-8))
            mr, vr = opt.state[param]["exp_avg"].numpy(), opt.state[param]["exp_avg_sq"].numpy()
            ok &= bool(np.allclose(m, mr, rtol=0, atol=1e-6 * np.abs(mr).max()))
            ok &= bool(np.allclose(v, vr, rtol=0, atol=1e-6 * np.abs(vr).max()))
    return ok


def pin_skip():
    rng = np.random.default_rng(3)
    p = (rng.standard_normal(16384) * 0.02).astype(np.float32)
    g = np.ones(16384, np.float32)
    g[3] = np.inf
    s, f = oracle.sumsq(g)
    p1, m1, v1 = p.copy(), np.zeros_like(p), np.zeros_like(p)
    _, _, skipped = oracle.step(oracle.make_hp(1e-3, 0.9, 0.95, 1e-8, 0.1, 1.0, 1.0, 1), s, f, g, p1, m1, v1)
    return skipped and np.array_equal(p1, p) and not m1.any()


def pin_e4m3():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    ours = oracle.e4m3_decode(codes)
    fin = ~np.isnan(ref)
    if not np.array_equal(ours[fin], ref[fin]):
        return False
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.uniform(-448, 448, 20000),
                        rng.standard_normal(20000) * 2.0 ** rng.integers(-12, 6, 20000)]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    if not np.array_equal(oracle.e4m3_encode(x), want):
        return False
    return all(int(oracle.e4m3_encode(np.array([np.float32(float(r[0]))]))[0]) == int(r[1], 16)
               for r in rows("e4m3_codes.txt"))


def pin_quantise():
    rng = np.random.default_rng(5)
    p = (rng.standard_normal(16384) * 0.02).astype(np.float32)
    q, s = oracle.quantise_block(p)
    amax = np.float32(np.abs(p).max())
    ok = s == amax / np.float32(448.0)
    ok &= oracle.quantise_block(np.zeros(16384, np.float32))[1] == 1.0
    ok &= int(q[int(np.argmax(np.abs(p)))]) in (0x7E, 0xFE)
    return bool(ok)


def pin_scaler():
    for n, s0, flags, scales, steps in rows("loss_scale_sequence.txt"):
        sc = oracle.Scaler(float(s0), int(n))
        got = []
        for fl in flags.split(","):
            sc.update(int(fl))
            got.append((sc.scale, sc.step))
        if got != list(zip([float(x) for x in scales.split(",")], [int(x) for x in steps.split(",")])):
            return False
    return True


def pin_mx():
    for v0, v1, v2, sc, c0, c1, c2 in rows("mx_group.txt"):
        g = np.array([float(v0), float(v1)] + [float(v2)] * 30, np.float32)
        q, s = oracle.mx_quantise(g)
        if int(s[0]) != int(sc) or [int(q[0]), int(q[1]), int(q[2])] != [int(c0, 16), int(c1, 16), int(c2, 16)]:
            return False
    e = torch.arange(0, 255, dtype=torch.uint8).view(torch.float8_e8m0fnu).float().numpy()
    return all(oracle.e8m0_decode(i) == e[i] for i in range(0, 255, 7))


def pin_split():
    for sizes, dp, owner, buckets, padded in rows("paramwise_split.txt"):
        o, b = oracle.paramwise_split([(1, int(x), 1) for x in sizes.split(",")], int(dp))
        if o.tolist() != [int(x) for x in owner.split(",")] or b.tolist() != [int(x) for x in buckets.split(",")]:
            return False
    return True


def pin_monitor():
    rng = np.random.default_rng(6)
    p = (rng.standard_normal(16384) * 0.02).astype(np.float32)
    p[:20] = 1e-9
    p[20] = 0.0
    q, s = oracle.quantise_block(p)
    c, u = oracle.quant_monitor(p, q, s)
    d = oracle.e4m3_decode(q).astype(np.float64) * s
    want = 1.0 - scipy_cosine_distance(p.astype(np.float64), d)
    return abs(c - want) < 1e-12 and u == int(np.sum((p != 0) & (oracle.e4m3_decode(q) == 0)))


PINS = [pin_fold, pin_layout, pin_sumsq, pin_clip_and_adamw, pin_skip, pin_e4m3, pin_quantise,
        pin_scaler, pin_mx, pin_split, pin_monitor]


def _run_pins():
    failed = []
    for pin in PINS:
        try:
            ok = pin()
        except AssertionError:
            ok = False
        if not ok:
            failed.append(pin.__name__)
    return failed


# ---------------------------------------------------------------------------
# the mistakes: (name, text in the oracle, replacement)

MUTATIONS = [
    ("no weight decay", "d.decay = (float)(1.0 - (double)hp->lr * (double)hp->weight_decay);",
     "d.decay = 1.0f;"),
    ("no bias correction of m", "double bc1 = 1.0 - pow((double)hp->beta1, t);", "double bc1 = 1.0;"),
    ("eps inside the square root", "float den = fmaf(sqrtf(vn), d->inv_sqrt_bc2, hp->eps);",
     "float den = sqrtf(vn * d->inv_sqrt_bc2 * d->inv_sqrt_bc2 + hp->eps);"),
    ("update sign", "float pn = fmaf(-d->step_size, mn / den, *p * d->decay);",
     "float pn = fmaf(d->step_size, mn / den, *p * d->decay);"),
    ("v from |g| not g^2", "float vn = fmaf(hp->beta2, *v, (d->omb2 * g) * g);",
     "float vn = fmaf(hp->beta2, *v, d->omb2 * fabsf(g));"),
    ("clip comparison flipped", "*clip_applies = coef < 1.0;", "*clip_applies = coef > 1.0;"),
    ("clip on the scaled norm", "double coef = (double)max_norm / (global + 1e-6);",
     "double coef = (double)max_norm / (scaled + 1e-6);"),
    ("scale = amax / 240", "float s = (amax == 0.0f) ? 1.0f : amax / 448.0f;",
     "float s = (amax == 0.0f) ? 1.0f : amax / 240.0f;"),
    ("E4M3 truncates", "float n = nearbyintf(ldexpf(a, 3 - e));", "float n = floorf(ldexpf(a, 3 - e));"),
    ("E4M3 overflow to NaN", "if (a >= 448.0f) return (uint8_t)(sign | 0x7E);",
     "if (a >= 448.0f) return (uint8_t)(sign | 0x7F);"),
    ("E4M3 drops the sign", "uint8_t sign = signbit(x) ? 0x80 : 0x00;", "uint8_t sign = 0x00;"),
    ("block order cb-major", "            for (int64_t rb = 0; rb < rbs; ++rb)\n                for (int64_t cb = 0; cb < cbs; ++cb) {",
     "            for (int64_t cb = 0; cb < cbs; ++cb)\n                for (int64_t rb = 0; rb < rbs; ++rb) {"),
    ("padding not zeroed", "                    memset(d, 0, (size_t)esz);", "                    memset(d, 0x11, (size_t)esz);"),
    ("shard size floored", "    int64_t per = ceil_div(nblk, dp);", "    int64_t per = nblk / dp;"),
    ("norm drops the last element", "for (int64_t i = 0; i < n; ++i) acc_add_square(a, g[i]);",
     "for (int64_t i = 0; i + 1 < n; ++i) acc_add_square(a, g[i]);"),
    ("inf not flagged", "        a->found_inf = 1;\n        if (mant) a->found_nan = 1;",
     "        if (mant) a->found_nan = 1;"),
    ("step not skipped", "    if (found_inf) return 1;\n    orc_derived d = derive(hp, sumsq);\n    for (int64_t k",
     "    if (0) return 1;\n    orc_derived d = derive(hp, sumsq);\n    for (int64_t k"),
    ("t advances on a skip", "        s->scale = s->scale * 0.5f;\n        s->good_steps = 0;",
     "        s->scale = s->scale * 0.5f;\n        s->step += 1;\n        s->good_steps = 0;"),
    ("MX scale exponent off by one", "        s = (k - 1) - 8;", "        s = k - 8;"),
    ("param-wise sort ascending", "            if (so >= sz) break;", "            if (so <= sz) break;"),
    ("underflow counts true zeros", "        if (p[i] != 0.0f && dq == 0.0) ++under;", "        if (dq == 0.0) ++under;"),
]


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


def test_unmodified_oracle_passes_every_pin():
    assert _run_pins() == []


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(source, name, old, new):
    assert source.count(old) == 1, f"mutation anchor not unique or missing: {name}"
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "mutant.c")
        so = os.path.join(d, "libmutant.so")
        with open(c, "w") as f:
            f.write(source.replace(old, new))
        subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", so, c, "-lm"],
                       check=True)
        with oracle.using_library(so):
            failed = _run_pins()
    assert failed, f"no pin caught: {name}"
