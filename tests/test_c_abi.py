"""The C ABI from plain C: tests/c_abi_example.c links libfp8z1.so and the
CUDA runtime only (no PyTorch, no Python binding) -- the boundary needs
nothing but pointers and sizes."""
import os
import subprocess

import numpy as np
import pytest

import oracle
from blockwise_fp8_zero_fold_gb300 import build as fp8build

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _cuda_home():
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and os.path.isdir(os.path.join(c, "include")):
            return c
    pytest.skip("no CUDA toolkit headers")


@pytest.fixture(scope="module")
def exe(tmp_path_factory):
    lib = fp8build.build()
    cuda = _cuda_home()
    out = str(tmp_path_factory.mktemp("cabi") / "c_abi_example")
    libdir = os.path.dirname(lib)
    subprocess.run(["gcc", "-std=c11", "-O2", "-Wall", "-o", out, os.path.join(HERE, "c_abi_example.c"),
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                    "-L", libdir, "-lfp8z1", "-Wl,-rpath," + libdir,
                    "-L", os.path.join(cuda, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(cuda, "lib64")],
                   check=True)
    return out


def test_host_calls_from_c(exe):
    out = subprocess.run([exe, "host"], capture_output=True, text=True, check=True).stdout.splitlines()
    shapes = [(1, 300, 200), (2, 129, 257)]
    nblk = oracle.count_blocks(shapes)
    assert out[0] == f"nblk {nblk} padded {nblk * 16384} real {300 * 200 + 2 * 129 * 257} " \
                     f"r0 {0} {oracle.shard_range(nblk, 2, 0)[1]} r1 {oracle.shard_range(nblk, 2, 1)[0]} {nblk}"
    p, e, rb, cb, rr, cr = oracle.build_lut(shapes)[5]
    assert out[1] == f"lut5 {p} {e} {rb} {cb} {rr} {cr}"
    o, b = oracle.paramwise_split(shapes, 2)
    assert out[2] == f"split {o[0]} {o[1]} {b[0]} {b[1]} {2 * max(b)}"
    assert out[3] == "scaler 32768 2"
    assert out[4] == "bad -1 invalid argument"


@pytest.mark.gpu
@pytest.mark.parametrize("mode,steps", [("gpu", 1), ("graph", 3), ("graph_patch", 3)])
def test_steps_from_c(exe, tmp_path, mode, steps):
    """One step, or three launches of one captured graph (t = 1, 2, 3 written
    to pinned memory between them, or patched into the executable graph's
    step node), from plain C against the oracle."""
    rng = np.random.default_rng(31)
    g = (rng.standard_normal((300, 200)) * 1024e-3).astype(np.float32)
    p = (rng.standard_normal((300, 200)) * 0.02).astype(np.float32)
    fin, fout = tmp_path / "in.bin", tmp_path / "out.bin"
    np.concatenate([g.ravel(), p.ravel()]).tofile(fin)
    r = subprocess.run([exe, mode, str(fin), str(fout)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    raw = np.fromfile(fout, dtype=np.uint8)
    n = 6 * 16384
    master = raw[:4 * n].view(np.float32)
    scales = raw[4 * n:4 * n + 24].view(np.float32)
    fp8 = raw[4 * n + 24:].reshape(300, 200)
    shapes = [(1, 300, 200)]
    og, op = oracle.fold(shapes, [g[None]]), oracle.fold(shapes, [p[None]])
    s, f = oracle.sumsq(og)
    om, ov = np.zeros_like(op), np.zeros_like(op)
    for t in range(1, steps + 1):
        q, sc, _ = oracle.step(oracle.make_hp(1e-3, 0.9, 0.95, 1e-8, 0.1, 1.0, 1024.0, t), s, f, og, op, om, ov)
    want = np.zeros((1, 300, 200), np.uint8)
    oracle.unfold(shapes, q, [want])
    assert np.array_equal(master.view(np.uint32), op.view(np.uint32))
    assert np.array_equal(scales, sc)
    assert np.array_equal(fp8, want[0])
