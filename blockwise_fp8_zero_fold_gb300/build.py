"""Build libfp8z1.so (and its checked variant) in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel into ``_build/<variant>/`` and
the objects are linked into ``blockwise_fp8_zero_fold_gb300/libfp8z1.so``.
The checked variant, ``libfp8z1_checked.so``, is the same sources compiled
with ``-DFP8Z1_CHECKED=1``: its kernels test every row-major param access
against the param's extent and skip and count the ones outside (a debug build
for the parity tests).  ``--fmad=false`` keeps the compiler from contracting
a*b+c: the kernels use explicit fused multiply-adds wherever the FP32 update
wants one.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libfp8z1.so")
LIB_CHECKED = os.path.join(PKG, "libfp8z1_checked.so")
SOURCES = ["layout.cpp", "fold.cu", "norm.cu", "step.cu", "step_full.cu", "step_pad.cu", "mx.cu"]
HEADERS = ["internal.h", "checked.cuh", "update.cuh", "step_args.h", "step_kernel.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def lib_path(checked: bool = False) -> str:
    return LIB_CHECKED if checked else LIB


def flags(verbose_ptxas: bool = False, checked: bool = False):
    f = ARCH + ["-lineinfo", "-O3", "--fmad=false", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                "-I", INCLUDE, "-I", CSRC]
    if checked:
        f += ["-DFP8Z1_CHECKED=1"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _stale(checked: bool) -> bool:
    lib = lib_path(checked)
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, s) for s in SOURCES + HEADERS] + [os.path.join(INCLUDE, "fp8z1.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def _build(variants, verbose_ptxas: bool = False):
    """Compile every source of every variant at once, then link each."""
    cc = nvcc()
    procs, objs = [], {}
    for checked in variants:
        out_dir = os.path.join(BUILD, "checked" if checked else "release")
        os.makedirs(out_dir, exist_ok=True)
        objs[checked] = []
        for s in SOURCES:
            obj = os.path.join(out_dir, s + ".o")
            objs[checked].append(obj)
            cmd = [cc] + flags(verbose_ptxas, checked) + ["-c", os.path.join(CSRC, s), "-o", obj]
            procs.append((s, checked, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for s, checked, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        tag = f"{s} (checked)" if checked else s
        if text.strip():
            sys.stderr.write(f"--- nvcc {tag}\n{text}")
        if p.returncode != 0:
            failed.append(tag)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    for checked in variants:
        lib = lib_path(checked)
        tmp = lib + f".tmp{os.getpid()}"
        subprocess.run([cc] + ARCH + ["-shared", "-o", tmp] + objs[checked], check=True)
        os.replace(tmp, lib)


def build(force: bool = False, verbose_ptxas: bool = False, checked: bool = False) -> str:
    """Build one variant (when stale or forced); returns its path."""
    if force or _stale(checked):
        _build([checked], verbose_ptxas)
    return lib_path(checked)


def build_all(force: bool = False, verbose_ptxas: bool = False):
    """Build the release and the checked library (the stale ones), together."""
    variants = [c for c in (False, True) if force or _stale(c)]
    if variants:
        _build(variants, verbose_ptxas)
    return [LIB, LIB_CHECKED]


if __name__ == "__main__":
    for p in build_all(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv):
        print(p)
