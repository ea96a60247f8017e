"""Host code under AddressSanitizer + UndefinedBehaviorSanitizer: the oracle
(every routine, compiled into tests/sanitize/oracle_driver.c) and the host
side of the C ABI (layout.cpp linked alone with
tests/sanitize/layout_driver.cpp, host-only layouts).  A sanitizer report
aborts the test program, failing the test."""
import os
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SAN = ["-O1", "-g", "-fsanitize=address,undefined", "-fno-sanitize-recover=all", "-fno-omit-frame-pointer"]


def _cuda_home():
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and os.path.isdir(os.path.join(c, "include")):
            return c
    pytest.skip("no CUDA toolkit headers")


def _build_and_run(cmd, exe):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0 and "sanitize" in r.stderr:
        pytest.skip("the compiler has no sanitizer runtime here")
    assert r.returncode == 0, r.stderr[-3000:]
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:abort_on_error=1",
               UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1")
    out = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=300)
    assert out.returncode == 0, (out.stdout + out.stderr)[-4000:]
    return out.stdout


def test_oracle_under_asan_ubsan(tmp_path):
    exe = str(tmp_path / "oracle_san")
    out = _build_and_run(["gcc", "-std=c11", "-ffp-contract=off", *SAN, os.path.join(HERE, "sanitize", "oracle_driver.c"),
                          "-o", exe, "-lm"], exe)
    assert "oracle driver ok" in out


def test_layout_builder_under_asan_ubsan(tmp_path):
    cuda = _cuda_home()
    exe = str(tmp_path / "layout_san")
    csrc = os.path.join(ROOT, "blockwise_fp8_zero_fold_gb300", "csrc")
    lib64 = os.path.join(cuda, "lib64")
    out = _build_and_run(["g++", "-std=c++17", *SAN, "-I", os.path.join(ROOT, "include"), "-I", csrc,
                          "-I", os.path.join(cuda, "include"), os.path.join(HERE, "sanitize", "layout_driver.cpp"),
                          os.path.join(csrc, "layout.cpp"), "-o", exe, "-L", lib64, "-lcudart",
                          "-Wl,-rpath," + lib64], exe)
    assert "layout driver ok" in out
