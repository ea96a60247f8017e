"""The allocation-free grad norm, fp8z1_grad_norm_noalloc.

It exists for callers that cannot call cudaMalloc (a framework whose caching
allocator owns the device memory, or a step loop that must not block on an
allocation); its workspace is a static device array.  This file is collected
last on purpose: each GPU test makes two calls in a row, so the second call
runs on the workspace the first one (or an earlier test) left behind.

Every result is checked against the oracle's exact sum of squares and inf
flag ("DeepSpeed ZeRO 优化" §七 / §六), within 1e-12 relative as built (the
bar is 1e-5), and against fp8z1_grad_norm, the layout-owned entry point."""
import numpy as np
import pytest
import torch

import oracle
from blockwise_fp8_zero_fold_gb300 import build as fp8build
from blockwise_fp8_zero_fold_gb300 import fp8z1 as F

B = F.BLOCK_ELEMS


def test_rejects_too_many_blocks_before_touching_the_device():
    fp8build.build()
    lib = F.lib()
    buf = np.zeros(64, np.float64)
    p = buf.ctypes.data
    assert lib.fp8z1_grad_norm_noalloc(p, F.NOALLOC_MAX_BLOCKS + 1, p, p, None) == F.EINVAL
    assert lib.fp8z1_grad_norm_noalloc(p, -1, p, p, None) == F.EINVAL
    assert lib.fp8z1_grad_norm_noalloc(None, 1, p, p, None) == F.EINVAL
    assert lib.fp8z1_grad_norm_noalloc(p + 4, 1, p, p, None) == F.EALIGN


def _pair():
    return (torch.zeros(1, dtype=torch.float64, device="cuda"),
            torch.zeros(1, dtype=torch.int32, device="cuda"))


def _close(got: float, want: float):
    assert abs(got - want) <= 1e-5 * want, (got, want)
    assert abs(got - want) <= 1e-12 * want, (got, want)


@pytest.mark.gpu
def test_matches_oracle_and_layout_grad_norm_on_two_calls_in_a_row():
    fp8build.build()
    assert torch.cuda.is_available()
    oracle.build()
    rng = np.random.default_rng(2024)
    nb_a, nb_b = 300, 37   # the second call runs fewer CTAs than the first
    L = F.fp8z1_build_layout([(nb_a, 128, 128)])
    a = (rng.standard_normal(nb_a * B) * 0.1).astype(np.float32)
    b = (rng.standard_normal(nb_b * B) * 3.0).astype(np.float32)
    b[12345] = np.inf
    da, db = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()

    ref_a, ref_b = _pair(), _pair()
    F.fp8z1_grad_norm(L, da, 0, nb_a, *ref_a)
    F.fp8z1_grad_norm(L, db, 0, nb_b, *ref_b)
    got_a, got_b = _pair(), _pair()
    F.fp8z1_grad_norm_noalloc(da, nb_a, *got_a)
    F.fp8z1_grad_norm_noalloc(db, nb_b, *got_b)
    torch.cuda.synchronize()
    exact_a, inf_a = oracle.sumsq(a)
    _, inf_b = oracle.sumsq(b)
    assert (inf_a, inf_b) == (0, 1)
    _close(got_a[0].item(), exact_a)
    _close(ref_a[0].item(), exact_a)
    assert got_a[1].item() == ref_a[1].item() == inf_a
    assert got_b[1].item() == ref_b[1].item() == inf_b
    # without the inf, the second call's sum is checked too
    b[12345] = 0.0
    db.copy_(torch.from_numpy(b))
    ref_b, got_b = _pair(), _pair()
    F.fp8z1_grad_norm(L, db, 0, nb_b, *ref_b)
    F.fp8z1_grad_norm_noalloc(db, nb_b, *got_b)
    torch.cuda.synchronize()
    exact_b, inf_b = oracle.sumsq(b)
    assert inf_b == 0
    _close(got_b[0].item(), exact_b)
    _close(ref_b[0].item(), exact_b)
    assert got_b[1].item() == 0


@pytest.mark.gpu
def test_at_the_block_limit_and_a_range_split_over_two_calls():
    """A call of exactly FP8Z1_NOALLOC_MAX_BLOCKS blocks (4.3 G grads, every
    CTA of the grid with many units), made twice in a row, then a range of the
    limit + 37 blocks split into two calls that accumulate into one sum."""
    fp8build.build()
    assert torch.cuda.is_available()
    oracle.build()
    torch.cuda.empty_cache()
    cap = F.NOALLOC_MAX_BLOCKS
    n = (cap + 37) * B
    g = torch.empty(n, dtype=torch.float32, device="cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(91)
    g.normal_(0.0, 1.0, generator=gen)
    g.mul_(1e-3 * 1024.0)     # loss-scaled grads, as the workloads store them
    g[7 * B + 5] = 250.0       # an outlier
    host = g.cpu().numpy()
    head, _ = oracle.sumsq_parallel([host[:cap * B]], threads=16)
    total, inf_total = oracle.sumsq_parallel([host], threads=16)
    assert inf_total == 0

    first, second = _pair(), _pair()
    F.fp8z1_grad_norm_noalloc(g, cap, *first)
    F.fp8z1_grad_norm_noalloc(g, cap, *second)
    torch.cuda.synchronize()
    _close(first[0].item(), head)
    assert second[0].item() == first[0].item()   # deterministic for a range
    assert first[1].item() == second[1].item() == 0

    split = _pair()   # the limit, then 37 more blocks: one accumulated sum
    F.fp8z1_grad_norm_noalloc(g, cap, *split)
    F.fp8z1_grad_norm_noalloc(g[cap * B:], 37, *split)
    torch.cuda.synchronize()
    _close(split[0].item(), total)
    assert split[1].item() == 0

    # the layout-owned entry point over the same range agrees
    L = F.fp8z1_build_layout([(cap + 37, 128, 128)])
    ref = _pair()
    F.fp8z1_grad_norm(L, g, 0, cap + 37, *ref)
    torch.cuda.synchronize()
    _close(ref[0].item(), total)
    assert abs(split[0].item() - ref[0].item()) <= 1e-12 * total
    del g, host
    torch.cuda.empty_cache()

