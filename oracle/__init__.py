"""fp8z1 oracle -- TEST INFRASTRUCTURE ONLY.

Python (ctypes + numpy) front of the plain single-threaded C oracle in
``fp8z1_oracle.c``.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package; the
CUDA library never does, and the two share no code.

Every function here is argument marshalling around the C oracle; the
arithmetic, with its citations, lives in the C file.

The shared library is compiled on first import (or when the C source is
newer) with ``gcc -std=c11 -O2 -ffp-contract=off``.
"""
from __future__ import annotations

import contextlib
import ctypes as C
import os
import subprocess
import threading
from typing import Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8z1_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_fp8z1.so")
_lock = threading.Lock()
_lib = None

TILE = 128
BLOCK_ELEMS = TILE * TILE


def build(force: bool = False) -> str:
    """Compile the oracle into ``liboracle_fp8z1.so`` (plain gcc, no CUDA)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-Wall",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


class Shape(C.Structure):
    _fields_ = [("E", C.c_int64), ("R", C.c_int64), ("C", C.c_int64)]


class Block(C.Structure):
    _fields_ = [("param", C.c_int64), ("expert", C.c_int64), ("row_block", C.c_int64),
                ("col_block", C.c_int64), ("rows_real", C.c_int64), ("cols_real", C.c_int64)]


class HP(C.Structure):
    _fields_ = [("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float),
                ("eps", C.c_float), ("weight_decay", C.c_float), ("max_norm", C.c_float),
                ("loss_scale", C.c_float), ("step", C.c_int64)]


class Acc(C.Structure):
    _fields_ = [("limb", C.c_uint64 * 10), ("found_inf", C.c_int32), ("found_nan", C.c_int32)]


class ScalerState(C.Structure):
    _fields_ = [("scale", C.c_float), ("step", C.c_int64), ("good_steps", C.c_int32),
                ("growth_interval", C.c_int32)]


def _bind(L):
    """Declare the C signatures on a loaded oracle library."""
    P = C.c_void_p
    i64, i32 = C.c_int64, C.c_int32
    L.oracle_count_blocks.argtypes = [C.POINTER(Shape), i32]
    L.oracle_count_blocks.restype = i64
    L.oracle_build_lut.argtypes = [C.POINTER(Shape), i32, C.POINTER(Block)]
    L.oracle_shard_range.argtypes = [i64, i32, i32, C.POINTER(i64), C.POINTER(i64)]
    L.oracle_fold.argtypes = [C.POINTER(Shape), i32, C.POINTER(P), P, i32, i64, i64]
    L.oracle_fold.restype = C.c_int
    L.oracle_unfold.argtypes = [C.POINTER(Shape), i32, P, C.POINTER(P), i32, i64, i64]
    L.oracle_unfold.restype = C.c_int
    L.oracle_acc_init.argtypes = [C.POINTER(Acc)]
    L.oracle_acc_add.argtypes = [C.POINTER(Acc), P, i64]
    L.oracle_acc_merge.argtypes = [C.POINTER(Acc), C.POINTER(Acc)]
    L.oracle_acc_result.argtypes = [C.POINTER(Acc)]
    L.oracle_acc_result.restype = C.c_double
    L.oracle_sumsq.argtypes = [P, i64, C.POINTER(C.c_double), C.POINTER(i32)]
    L.oracle_clip_coef.argtypes = [C.c_double, C.c_float, C.c_float,
                                   C.POINTER(C.c_double), C.POINTER(C.c_double),
                                   C.POINTER(i32)]
    L.oracle_e4m3_encode.argtypes = [C.c_float]
    L.oracle_e4m3_encode.restype = C.c_uint8
    L.oracle_e4m3_decode.argtypes = [C.c_uint8]
    L.oracle_e4m3_decode.restype = C.c_float
    L.oracle_e4m3_encode_n.argtypes = [P, P, i64]
    L.oracle_e4m3_decode_n.argtypes = [P, P, i64]
    L.oracle_quantise_block.argtypes = [P, P, C.POINTER(C.c_float)]
    L.oracle_step.argtypes = [C.POINTER(HP), C.c_double, i32, P, P, P, P, P, P, i64]
    L.oracle_step.restype = C.c_int
    L.oracle_scaler_update.argtypes = [C.POINTER(ScalerState), i32]
    L.oracle_paramwise_split.argtypes = [C.POINTER(Shape), i32, i32, P, P]
    L.oracle_quant_monitor.argtypes = [P, P, C.c_float, i64, C.POINTER(C.c_double),
                                       C.POINTER(i64)]
    L.oracle_e8m0_decode.argtypes = [C.c_uint8]
    L.oracle_e8m0_decode.restype = C.c_float
    L.oracle_mx_quantise_group.argtypes = [P, P, P]
    L.oracle_mx_step.argtypes = [C.POINTER(HP), C.c_double, i32, P, P, P, P, P, P, i64]
    L.oracle_mx_step.restype = C.c_int
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(C.CDLL(_LIB))
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Run this front against another build of the oracle for a while (the
    tests use it to plant mistakes in a copy and check that the pins fail)."""
    global _lib
    lib()
    with _lock:
        old = _lib
        _lib = _bind(C.CDLL(path))
    try:
        yield
    finally:
        with _lock:
            _lib = old


# ---------------------------------------------------------------------------
# helpers

def _shapes(shapes: Sequence[Sequence[int]]):
    arr = (Shape * max(1, len(shapes)))()
    for i, s in enumerate(shapes):
        if len(s) == 2:
            e, r, c = 1, s[0], s[1]
        else:
            e, r, c = s
        arr[i] = Shape(int(e), int(r), int(c))
    return arr, len(shapes)


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle wants C-contiguous arrays"
    return a.ctypes.data


# ---------------------------------------------------------------------------
# layout

def count_blocks(shapes) -> int:
    arr, n = _shapes(shapes)
    return int(lib().oracle_count_blocks(arr, n))


def build_lut(shapes) -> np.ndarray:
    """int64 array [nblk, 6]: param, expert, row_block, col_block, rows_real, cols_real."""
    arr, n = _shapes(shapes)
    nblk = count_blocks(shapes)
    out = (Block * max(1, nblk))()
    lib().oracle_build_lut(arr, n, out)
    return np.ctypeslib.as_array(C.cast(out, C.POINTER(C.c_int64)), shape=(max(1, nblk), 6))[:nblk].copy()


def shard_range(nblk: int, dp: int, rank: int):
    b0, b1 = C.c_int64(), C.c_int64()
    lib().oracle_shard_range(int(nblk), int(dp), int(rank), C.byref(b0), C.byref(b1))
    return b0.value, b1.value


def fold(shapes, srcs: Sequence[np.ndarray], b0: int = 0, b1: int | None = None) -> np.ndarray:
    """Fold row-major params (numpy arrays, 1/2/4-byte dtype) into blocks [b0, b1)."""
    arr, n = _shapes(shapes)
    if b1 is None:
        b1 = count_blocks(shapes)
    dtype = srcs[0].dtype
    assert all(s.dtype == dtype for s in srcs)
    ptrs = (C.c_void_p * max(1, n))(*[_ptr(s) for s in srcs])
    out = np.empty((b1 - b0) * BLOCK_ELEMS, dtype=dtype)
    rc = lib().oracle_fold(arr, n, ptrs, out.ctypes.data, dtype.itemsize, b0, b1)
    assert rc == 0
    return out


def unfold(shapes, src: np.ndarray, dsts: Sequence[np.ndarray], b0: int = 0, b1: int | None = None):
    """Unfold blocks [b0, b1) of ``src`` into the row-major arrays ``dsts`` (in place)."""
    arr, n = _shapes(shapes)
    if b1 is None:
        b1 = count_blocks(shapes)
    assert src.size == (b1 - b0) * BLOCK_ELEMS
    ptrs = (C.c_void_p * max(1, n))(*[_ptr(d) for d in dsts])
    rc = lib().oracle_unfold(arr, n, _ptr(src), ptrs, src.dtype.itemsize, b0, b1)
    assert rc == 0


# ---------------------------------------------------------------------------
# norm

class SumsqAccumulator:
    """Exact sum of squares of float32 chunks; result() rounds once to double."""

    def __init__(self):
        self._a = Acc()
        lib().oracle_acc_init(C.byref(self._a))

    def add(self, g: np.ndarray):
        g = np.ascontiguousarray(g, dtype=np.float32)
        lib().oracle_acc_add(C.byref(self._a), g.ctypes.data, g.size)

    def merge(self, other: "SumsqAccumulator"):
        lib().oracle_acc_merge(C.byref(self._a), C.byref(other._a))

    def result(self) -> float:
        return float(lib().oracle_acc_result(C.byref(self._a)))

    @property
    def found_inf(self) -> int:
        return int(self._a.found_inf)


def sumsq_parallel(arrays, threads: int = 8, chunk: int = 1 << 24):
    """Exact sum of squares of several float32 arrays, chunks added in threads
    (each chunk through the same single-threaded accumulator, then merged
    exactly).  Returns (sumsq, found_inf)."""
    from concurrent.futures import ThreadPoolExecutor
    pieces = []
    for a in arrays:
        a = np.ascontiguousarray(a, dtype=np.float32).reshape(-1)
        for i in range(0, a.size, chunk):
            pieces.append(a[i:i + chunk])

    def work(p):
        acc = SumsqAccumulator()
        acc.add(p)
        return acc

    total = SumsqAccumulator()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        for acc in ex.map(work, pieces):
            total.merge(acc)
    return total.result(), total.found_inf


def sumsq(g: np.ndarray):
    g = np.ascontiguousarray(g, dtype=np.float32)
    s, f = C.c_double(), C.c_int32()
    lib().oracle_sumsq(g.ctypes.data, g.size, C.byref(s), C.byref(f))
    return s.value, f.value


def clip_coef(sumsq_value: float, max_norm: float, loss_scale: float):
    """(global_norm, clip_coef, clip_applies) in double."""
    gn, cc, ap = C.c_double(), C.c_double(), C.c_int32()
    lib().oracle_clip_coef(float(sumsq_value), float(max_norm), float(loss_scale),
                           C.byref(gn), C.byref(cc), C.byref(ap))
    return gn.value, cc.value, bool(ap.value)


# ---------------------------------------------------------------------------
# E4M3

def e4m3_encode(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    q = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode_n(x.ctypes.data, q.ctypes.data, x.size)
    return q


def e4m3_decode(q: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    x = np.empty(q.shape, dtype=np.float32)
    lib().oracle_e4m3_decode_n(q.ctypes.data, x.ctypes.data, q.size)
    return x


def quantise_block(p: np.ndarray):
    p = np.ascontiguousarray(p, dtype=np.float32)
    assert p.size == BLOCK_ELEMS
    q = np.empty(BLOCK_ELEMS, dtype=np.uint8)
    s = C.c_float()
    lib().oracle_quantise_block(p.ctypes.data, q.ctypes.data, C.byref(s))
    return q, s.value


# ---------------------------------------------------------------------------
# step

def make_hp(lr, beta1, beta2, eps, weight_decay, max_norm, loss_scale, step) -> HP:
    return HP(lr, beta1, beta2, eps, weight_decay, max_norm, loss_scale, int(step))


def step(hp: HP, sumsq_value: float, found_inf: int, grad: np.ndarray, master: np.ndarray,
         m: np.ndarray, v: np.ndarray):
    """AdamW + quantise over folded blocks; master/m/v updated in place.

    Returns (codes uint8[n], scales float32[nblocks], skipped)."""
    n = grad.size
    assert n % BLOCK_ELEMS == 0
    for a in (grad, master, m, v):
        assert a.dtype == np.float32 and a.size == n and a.flags["C_CONTIGUOUS"]
    nb = n // BLOCK_ELEMS
    codes = np.zeros(n, dtype=np.uint8)
    scales = np.zeros(nb, dtype=np.float32)
    skipped = lib().oracle_step(C.byref(hp), float(sumsq_value), int(found_inf), grad.ctypes.data,
                                master.ctypes.data, m.ctypes.data, v.ctypes.data,
                                codes.ctypes.data, scales.ctypes.data, nb)
    return codes, scales, bool(skipped)


# ---------------------------------------------------------------------------
# loss scaler

class Scaler:
    def __init__(self, scale: float, growth_interval: int, step: int = 0):
        self.s = ScalerState(scale, step, 0, growth_interval)

    def update(self, found_inf: int):
        lib().oracle_scaler_update(C.byref(self.s), int(found_inf))

    @property
    def scale(self):
        return self.s.scale

    @property
    def step(self):
        return self.s.step

    @property
    def good_steps(self):
        return self.s.good_steps


# ---------------------------------------------------------------------------
# param-wise split, quantisation monitors, MXFP8

def paramwise_split(shapes, dp: int):
    """(owner[n], bucket_elems[dp]) of the greedy param-wise split."""
    arr, n = _shapes(shapes)
    owner = np.zeros(max(1, n), np.int32)
    bucket = np.zeros(max(1, dp), np.int64)
    lib().oracle_paramwise_split(arr, n, int(dp), owner.ctypes.data, bucket.ctypes.data)
    return owner[:n], bucket[:dp]


def quant_monitor(p: np.ndarray, q: np.ndarray, scale: float):
    """(cosine, underflow count) of one block."""
    p = np.ascontiguousarray(p, dtype=np.float32)
    q = np.ascontiguousarray(q, dtype=np.uint8)
    assert p.size == q.size
    c, u = C.c_double(), C.c_int64()
    lib().oracle_quant_monitor(p.ctypes.data, q.ctypes.data, float(scale), p.size, C.byref(c), C.byref(u))
    return c.value, u.value


MX_GROUP = 32


def e8m0_decode(e: int) -> float:
    return float(lib().oracle_e8m0_decode(int(e)))


def mx_quantise(p: np.ndarray):
    """Codes and E8M0 scale codes of consecutive groups of 32 values."""
    p = np.ascontiguousarray(p, dtype=np.float32).reshape(-1)
    assert p.size % MX_GROUP == 0
    q = np.empty(p.size, np.uint8)
    sc = np.empty(p.size // MX_GROUP, np.uint8)
    for g in range(sc.size):
        lib().oracle_mx_quantise_group(p[g * 32:].ctypes.data, q[g * 32:].ctypes.data,
                                       sc[g:].ctypes.data)
    return q, sc


def mx_step(hp: HP, sumsq_value: float, found_inf: int, grad, master, m, v):
    """AdamW + MXFP8 quantise over flat groups of 32; master/m/v in place.
    Returns (codes uint8[n], E8M0 scale codes uint8[n/32], skipped)."""
    n = grad.size
    assert n % MX_GROUP == 0
    for a in (grad, master, m, v):
        assert a.dtype == np.float32 and a.size == n and a.flags["C_CONTIGUOUS"]
    codes = np.zeros(n, np.uint8)
    scales = np.zeros(n // MX_GROUP, np.uint8)
    skipped = lib().oracle_mx_step(C.byref(hp), float(sumsq_value), int(found_inf), grad.ctypes.data,
                                   master.ctypes.data, m.ctypes.data, v.ctypes.data,
                                   codes.ctypes.data, scales.ctypes.data, n // MX_GROUP)
    return codes, scales, bool(skipped)
