"""Empty block (or group) ranges: every entry point that takes a range
enqueues nothing for b0 == b1 and leaves every buffer as it was.

An empty range is what the last DP rank gets when D does not divide the
block count ("面向 Blockwise FP8 量化的 ZeRO 优化器设计" §块粒度切分: each rank
holds a contiguous range of ceil(nblk / D) blocks, the last ranks fewer or
none); the range itself is checked against the oracle's shard arithmetic."""
import pytest
import torch

import oracle
from blockwise_fp8_zero_fold_gb300 import build as fp8build
from blockwise_fp8_zero_fold_gb300 import fp8z1 as F

B = F.BLOCK_ELEMS
SHAPES = [(1, 300, 200)]  # 3 x 2 = 6 blocks; D = 4 gives ranks of 2, 2, 2, 0 blocks
DP = 4


@pytest.fixture(scope="module")
def lib():
    fp8build.build()
    assert torch.cuda.is_available()
    oracle.build()
    return F.lib()


def _sentinel(n, dtype, value):
    return torch.full((n,), value, dtype=dtype, device="cuda")


@pytest.mark.gpu
def test_every_range_entry_point_enqueues_nothing_on_an_empty_range(lib):
    L = F.fp8z1_build_layout(SHAPES, DP)
    nblk = F.fp8z1_layout_info(L)[0]
    b0, b1 = F.fp8z1_shard_range(L, DP - 1)
    assert (b0, b1) == oracle.shard_range(nblk, DP, DP - 1) == (nblk, nblk)
    n = nblk * B
    bufs = {
        "grad": _sentinel(n, torch.float32, 7.0), "master": _sentinel(n, torch.float32, 1.5),
        "m": _sentinel(n, torch.float32, 2.5), "v": _sentinel(n, torch.float32, 3.5),
        "codes": _sentinel(n, torch.uint8, 0x5A), "scales": _sentinel(nblk, torch.float32, 9.0),
        "cos": _sentinel(nblk, torch.float32, -2.0), "under": _sentinel(nblk, torch.int32, 77),
        "sumsq": _sentinel(1, torch.float64, 11.0), "found": _sentinel(1, torch.int32, 0),
        "sel": _sentinel(1, torch.int32, 0),
    }
    grads = [_sentinel(300 * 200, torch.float32, 4.0).view(1, 300, 200)]
    fp8 = [_sentinel(300 * 200, torch.uint8, 0xA5).view(1, 300, 200)]
    gptrs = torch.tensor([t.data_ptr() for t in grads], dtype=torch.int64, device="cuda")
    fptrs = torch.tensor([t.data_ptr() for t in fp8], dtype=torch.int64, device="cuda")
    before = {k: v.clone() for k, v in bufs.items()}
    before_g, before_f = grads[0].clone(), fp8[0].clone()
    hp = F.make_hp(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=1.0,
                   loss_scale=1024.0, step=1)
    common = dict(master_shard=bufs["master"], m_shard=bufs["m"], v_shard=bufs["v"],
                  scale_shard=bufs["scales"], d_sumsq=bufs["sumsq"], d_found_inf=bufs["found"])
    torch.cuda.synchronize()
    for r0 in (b0, 2):  # the last rank's empty range, and an empty range inside the buffer
        n0 = F.fp8z1_kernel_launches()
        F.fp8z1_fold(L, gptrs, bufs["grad"], 4, r0, r0)
        F.fp8z1_unfold(L, bufs["codes"], fptrs, 1, r0, r0)
        F.fp8z1_grad_norm(L, bufs["grad"], r0, r0, bufs["sumsq"], bufs["found"])
        F.fp8z1_fold_norm(L, gptrs, None, r0, r0, bufs["sumsq"], bufs["found"])
        F.fp8z1_fold_norm(L, gptrs, bufs["grad"], r0, r0, bufs["sumsq"], bufs["found"])
        F.fp8z1_step(L, hp, bufs["grad"], bufs["master"], bufs["m"], bufs["v"], bufs["codes"],
                     bufs["scales"], r0, r0, bufs["sumsq"], bufs["found"])
        F.fp8z1_step_fused(L, hp, d_grad_params=gptrs, d_fp8_params=fptrs, b0=r0, b1=r0, **common)
        F.fp8z1_step_fused(L, hp, grad_shard=bufs["grad"], fp8_shard=bufs["codes"], block_cos=bufs["cos"],
                           block_underflow=bufs["under"], b0=r0, b1=r0, **common)
        F.fp8z1_step_fused_select(L, hp, hp, bufs["sel"], d_grad_params=gptrs, d_fp8_params=fptrs,
                                  b0=r0, b1=r0, **common)
        torch.cuda.synchronize()
        assert F.fp8z1_kernel_launches() == n0
        for k, v in bufs.items():
            assert torch.equal(v, before[k]), k
        assert torch.equal(grads[0], before_g) and torch.equal(fp8[0], before_f)
    assert F.fp8z1_device_status(L) == 0


@pytest.mark.gpu
def test_mx_entry_points_enqueue_nothing_on_an_empty_group_range(lib):
    shapes = [(1, 64, 96)]  # 192 groups of 32
    L = F.fp8z1_mx_build_layout(shapes, 1)
    groups, n = F.fp8z1_mx_layout_info(L)
    assert (groups, n) == (64 * 96 // 32, 64 * 96)
    bufs = {
        "grad": _sentinel(n, torch.float32, 7.0), "master": _sentinel(n, torch.float32, 1.5),
        "m": _sentinel(n, torch.float32, 2.5), "v": _sentinel(n, torch.float32, 3.5),
        "codes": _sentinel(n, torch.uint8, 0x5A), "scales": _sentinel(groups, torch.uint8, 0x33),
        "sumsq": _sentinel(1, torch.float64, 11.0), "found": _sentinel(1, torch.int32, 0),
        "sel": _sentinel(1, torch.int32, 1),
    }
    before = {k: v.clone() for k, v in bufs.items()}
    hp = F.make_hp(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=1.0,
                   loss_scale=1024.0, step=1)
    torch.cuda.synchronize()
    for g0 in (0, 64, groups):
        n0 = F.fp8z1_kernel_launches()
        F.fp8z1_mx_grad_norm(L, bufs["grad"], g0, g0, bufs["sumsq"], bufs["found"])
        F.fp8z1_mx_step(L, hp, bufs["grad"], bufs["master"], bufs["m"], bufs["v"], bufs["codes"],
                        bufs["scales"], g0, g0, bufs["sumsq"], bufs["found"])
        F.fp8z1_mx_step_select(L, hp, hp, bufs["sel"], bufs["grad"], bufs["master"], bufs["m"], bufs["v"],
                               bufs["codes"], bufs["scales"], g0, g0, bufs["sumsq"], bufs["found"])
        torch.cuda.synchronize()
        assert F.fp8z1_kernel_launches() == n0
        for k, v in bufs.items():
            assert torch.equal(v, before[k]), k
