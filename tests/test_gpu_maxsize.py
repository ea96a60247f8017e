"""One weight of more than 2^31 elements (46341 x 46341, 131 769 blocks):
every row-major offset past 2^31 must be formed in 64 bits, in the flat-run
norm, the step's fused fold of the grads and unfold of the codes.  One fused
step with clipping off; the norm against the oracle's exact sum, and sampled
blocks -- among them the last rows, past element 2^31 -- against the oracle
run on those blocks alone (blocks are independent once the global sum of
squares is fixed, "面向 Blockwise FP8 量化的 ZeRO 优化器设计" §总结)."""
import numpy as np
import pytest
import torch

import oracle
from blockwise_fp8_zero_fold_gb300 import fp8z1 as F
from blockwise_fp8_zero_fold_gb300.optimizer import ShardOptimizer
from tests._gpu import lib, to_host  # noqa: F401

pytestmark = pytest.mark.gpu
B = 16384
N = 46341  # N * N > 2**31
HP = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=1e30)


def test_weight_past_2_to_31_elements(lib):
    assert N * N > 2**31
    shape = (1, N, N)
    gen = torch.Generator(device="cuda").manual_seed(77)
    opt = ShardOptimizer([shape], loss_scale=1024.0, **HP)
    nb = -(-N // 128)
    assert opt.nblk == nb * nb
    master = torch.empty(shape, device="cuda").normal_(0, 0.02, generator=gen)
    opt.init_state([master])
    g = torch.empty(shape, device="cuda").normal_(0, 1.0, generator=gen)
    fp8 = torch.full(shape, 0x7F, dtype=torch.uint8, device="cuda")  # the NaN code: never written
    assert opt.step([g], [fp8]) == 0
    torch.cuda.synchronize()
    got_sumsq = float(opt.sumsq.item())
    gh = to_host(g).reshape(-1)
    exact, fi = oracle.sumsq_parallel([gh], threads=16)
    assert fi == 0 and abs(got_sumsq - exact) <= 1e-12 * exact

    hp = oracle.make_hp(loss_scale=1024.0, step=1, **HP)
    mh = to_host(master)[0]
    g2 = gh.reshape(N, N)
    reached = False
    for rb, cb in [(0, 0), (181, 181), (362, 0), (362, 181), (362, 362), (361, 362)]:
        k = rb * nb + cb
        r0, c0 = 128 * rb, 128 * cb
        rr, cr = min(128, N - r0), min(128, N - c0)
        tile = [(1, rr, cr)]
        ob_g = oracle.fold(tile, [np.ascontiguousarray(g2[r0:r0 + rr, c0:c0 + cr])[None]])
        ob_p = oracle.fold(tile, [np.ascontiguousarray(mh[r0:r0 + rr, c0:c0 + cr])[None]])
        om, ov = np.zeros_like(ob_p), np.zeros_like(ob_p)
        q, sc, _ = oracle.step(hp, got_sumsq, 0, ob_g, ob_p, om, ov)
        assert np.array_equal(to_host(opt.master[k * B:(k + 1) * B]).view(np.uint32), ob_p.view(np.uint32))
        assert np.array_equal(to_host(opt.v[k * B:(k + 1) * B]).view(np.uint32), ov.view(np.uint32))
        assert float(opt.scales[k]) == float(sc[0])
        want = np.zeros((1, rr, cr), np.uint8)
        oracle.unfold(tile, q, [want])
        assert np.array_equal(to_host(fp8[0, r0:r0 + rr, c0:c0 + cr]), want[0])
        reached |= (r0 + rr - 1) * N + (c0 + cr - 1) >= 2**31
    assert reached  # a sampled block lies past element 2^31
    assert not (fp8 == 0x7F).any()  # every element got its code
    assert F.fp8z1_device_status(opt.layout) == 0
