"""The allocation-free grad norm, fp8z1_grad_norm_noalloc.

It exists for callers that cannot call cudaMalloc (a framework whose caching
allocator owns the device memory, or a step loop that must not block on an
allocation); its workspace is a static device array.  This file is collected
last on purpose: the GPU test checks the call against fp8z1_grad_norm on two
calls in a row, so the second call runs on the workspace the first one left
behind."""
import ctypes as C

import numpy as np
import pytest
import torch

from blockwise_fp8_zero_fold_gb300 import build as fp8build
from blockwise_fp8_zero_fold_gb300 import fp8z1 as F


def test_rejects_too_many_blocks_before_touching_the_device():
    fp8build.build()
    lib = F.lib()
    buf = np.zeros(64, np.float64)
    p = buf.ctypes.data
    assert lib.fp8z1_grad_norm_noalloc(p, F.NOALLOC_MAX_BLOCKS + 1, p, p, None) == F.EINVAL
    assert lib.fp8z1_grad_norm_noalloc(p, -1, p, p, None) == F.EINVAL
    assert lib.fp8z1_grad_norm_noalloc(None, 1, p, p, None) == F.EINVAL
    assert lib.fp8z1_grad_norm_noalloc(p + 4, 1, p, p, None) == F.EALIGN


@pytest.mark.gpu
def test_matches_layout_grad_norm_on_two_calls_in_a_row():
    fp8build.build()
    assert torch.cuda.is_available()
    rng = np.random.default_rng(2024)
    nb_a, nb_b = 300, 37   # the second call uses fewer CTAs than the first
    L = F.fp8z1_build_layout([(nb_a, 128, 128)])
    a = (rng.standard_normal(nb_a * 16384) * 0.1).astype(np.float32)
    b = (rng.standard_normal(nb_b * 16384) * 3.0).astype(np.float32)
    b[12345] = np.inf
    da, db = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()

    def pair():
        return (torch.zeros(1, dtype=torch.float64, device="cuda"),
                torch.zeros(1, dtype=torch.int32, device="cuda"))

    ref_a, ref_b = pair(), pair()
    F.fp8z1_grad_norm(L, da, 0, nb_a, *ref_a)
    F.fp8z1_grad_norm(L, db, 0, nb_b, *ref_b)
    got_a, got_b = pair(), pair()
    F.fp8z1_grad_norm_noalloc(da, nb_a, *got_a)
    F.fp8z1_grad_norm_noalloc(db, nb_b, *got_b)
    torch.cuda.synchronize()
    sa, sb = ref_a[0].item(), got_a[0].item()
    assert abs(sb - sa) <= 1e-12 * sa, (sa, sb)
    assert got_a[1].item() == ref_a[1].item() == 0
    assert got_b[1].item() == ref_b[1].item() == 1
    # without the inf, the second call's sum is checked too
    b[12345] = 0.0
    db.copy_(torch.from_numpy(b))
    ref_b, got_b = pair(), pair()
    F.fp8z1_grad_norm(L, db, 0, nb_b, *ref_b)
    F.fp8z1_grad_norm_noalloc(db, nb_b, *got_b)
    torch.cuda.synchronize()
    s1, s2 = ref_b[0].item(), got_b[0].item()
    assert abs(s2 - s1) <= 1e-12 * s1, (s1, s2)
    assert got_b[1].item() == 0
