"""The checked build (libfp8z1_checked.so): the parity tests rerun on it with
no row-major access outside a param, and its checks fire where a table entry
points outside one.

The checked kernels test each load and store they make to a row-major param
against the param's extent, skip the ones outside and count them
(fp8z1_checked_misses).  A device memory checker is not available here; this
build stands in for one on the accesses the block table and the run tables
steer."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from blockwise_fp8_zero_fold_gb300 import build as fp8build
from blockwise_fp8_zero_fold_gb300 import fp8z1 as F
from tests._gpu import lib, to_host  # noqa: F401

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# every GPU test file that drives the library through Python (the maximum-size
# one included: a weight past 2^31 elements, where offsets need 64 bits),
# minus the ones that run the bench or link the library from C, and the
# literal ragged workload (160 GB on the device; the small-block file covers
# its block shapes)
SUITES = ["test_gpu_fold.py", "test_gpu_norm.py", "test_gpu_step.py", "test_gpu_fused.py", "test_gpu_next.py",
          "test_gpu_graph.py", "test_gpu_resume.py", "test_gpu_workloads.py", "test_gpu_maxsize.py",
          "test_gpu_random_layouts.py", "test_gpu_small_blocks.py", "test_zz_no_alloc.py"]


def test_parity_suites_on_the_checked_build(lib):
    if F.CHECKED:
        pytest.skip("runs the checked build from the release one")
    fp8build.build(checked=True)
    env = dict(os.environ, FP8Z1_CHECKED="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider"] + \
        [os.path.join("tests", s) for s in SUITES] + \
        ["tests/test_gpu_checked.py::test_checked_kernels_skip_and_count"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and " failed" not in r.stdout


@pytest.mark.plants_miss
def test_checked_kernels_skip_and_count(lib):
    """Block 0's device table entry is moved to start where its param ends.
    The three params sit back to back in one allocation, so the moved tile
    lies inside param 1's memory: an unchecked kernel would read or overwrite
    param 1 there (never memory outside the allocation).  The checked kernels
    skip every such access and count it, and leave param 1 alone."""
    if not F.CHECKED:
        pytest.skip("needs the checked build (FP8Z1_CHECKED=1)")
    shapes = [(1, 128, 128)] * 3
    L = F.fp8z1_build_layout(shapes)
    n = 16384
    rng = np.random.default_rng(21)
    g = torch.from_numpy(rng.standard_normal(3 * n).astype(np.float32)).cuda()
    gparams = [g[i * n:(i + 1) * n] for i in range(3)]
    gptrs = F.param_pointers(gparams)
    lut = F.fp8z1_copy_lut(L)
    entry = F.fp8z1_block(*[int(lut[0][f]) for f in ("src_offset", "param", "expert", "row_block",
                                                        "col_block", "ld", "rows_real", "cols_real")])
    entry.src_offset = n  # one past param 0's last element
    F.fp8z1_checked_set_lut_entry(L, 0, entry)

    # fold: block 0's 128 x 32 float4 loads are skipped (zeros), blocks 1-2 folded
    m0 = F.fp8z1_checked_misses()
    shard = torch.full((3 * n,), 7.0, device="cuda")
    F.fp8z1_fold(L, gptrs, shard, 4, 0, 3)
    m1 = F.fp8z1_checked_misses()
    assert m1 - m0 == 128 * 32
    host = to_host(shard)
    assert (host[:n] == 0).all()
    assert np.array_equal(host[n:], to_host(g)[n:])

    # unfold of 1-byte codes: block 0's 128 x 8 stores of 16 bytes are skipped
    codes = torch.from_numpy(rng.integers(0, 256, 3 * n, dtype=np.uint8)).cuda()
    out = torch.full((3 * n,), 0x3C, dtype=torch.uint8, device="cuda")
    F.fp8z1_unfold(L, codes, F.param_pointers([out[i * n:(i + 1) * n] for i in range(3)]), 1, 0, 3)
    m2 = F.fp8z1_checked_misses()
    assert m2 - m1 == 128 * 8
    ho = to_host(out)
    assert (ho[:n] == 0x3C).all()  # param 0 untouched
    assert np.array_equal(ho[n:], to_host(codes)[n:])  # param 1 holds only block 1's codes

    # the fold fused with the norm (with store: every block through the table)
    s = torch.zeros(1, dtype=torch.float64, device="cuda")
    f = torch.zeros(1, dtype=torch.int32, device="cuda")
    shard2 = torch.empty(3 * n, device="cuda")
    F.fp8z1_fold_norm(L, gptrs, shard2, 0, 3, s, f)
    m3 = F.fp8z1_checked_misses()
    assert m3 - m2 == 2 * 256 * 8  # two 64-row units of 256 threads x 8 float4
    gh = to_host(g).astype(np.float64)
    assert abs(s.item() - float((gh[n:] ** 2).sum())) <= 1e-9 * float((gh[n:] ** 2).sum())

    # the fused step: block 0's 512 x 8 grad loads and 512 x 8 code stores
    master = torch.from_numpy(rng.standard_normal(3 * n).astype(np.float32) * 0.02).cuda()
    mom1 = torch.zeros(3 * n, device="cuda")
    mom2 = torch.zeros(3 * n, device="cuda")
    scales = torch.zeros(3, device="cuda")
    hp = F.make_hp(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_norm=1.0,
                   loss_scale=1.0, step=1)
    out2 = torch.full((3 * n,), 0x3C, dtype=torch.uint8, device="cuda")
    F.fp8z1_step_fused(L, hp, d_grad_params=gptrs, master_shard=master, m_shard=mom1, v_shard=mom2,
                       d_fp8_params=F.param_pointers([out2[i * n:(i + 1) * n] for i in range(3)]),
                       scale_shard=scales, b0=0, b1=3, d_sumsq=s, d_found_inf=f)
    m4 = F.fp8z1_checked_misses()
    assert m4 - m3 == 2 * 512 * 8
    assert (to_host(out2)[:n] == 0x3C).all()
    assert F.fp8z1_device_status(L) == 0
