"""ctypes binding of libfp8z1.so: the same entry points, same names.

Argument marshalling only -- every step of the path runs in the library's
CUDA kernels.  Tensors (torch) are passed by ``data_ptr()``; plain ints are
taken as raw pointers.  ``stream`` is a ``torch.cuda.Stream``, a raw
``cudaStream_t`` int, or None for torch's current stream.  A non-zero status
raises ``Fp8z1Error``.  The library must have been built
(``__graft_entry__.build()``); there is no fallback.

With ``FP8Z1_CHECKED=1`` in the environment the checked build,
``libfp8z1_checked.so``, is loaded instead: the same entry points, with every
row-major param access of its kernels tested against the param's extent
(``fp8z1_checked_misses`` counts the ones skipped).
"""
from __future__ import annotations

import ctypes as C
import os
import threading
from typing import Sequence

import numpy as np

CHECKED = os.environ.get("FP8Z1_CHECKED", "0") not in ("", "0")
_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                         "libfp8z1_checked.so" if CHECKED else "libfp8z1.so")
_lock = threading.Lock()
_lib = None

BLOCK_ELEMS = 16384
MX_GROUP = 32
TILE = 128
LAYOUT_HOST_ONLY = 1
DEVSTATUS_BADPTR = 1
BUILD_CHECKED = 1

OK, EINVAL, EALIGN, ENOMEM, ECUDA, ENODEV = 0, -1, -2, -3, -4, -5


class Fp8z1Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fp8z1_strerror(status)} ({status})")


class fp8z1_shape(C.Structure):
    _fields_ = [("E", C.c_int64), ("R", C.c_int64), ("C", C.c_int64)]


class fp8z1_block(C.Structure):
    _fields_ = [("src_offset", C.c_int64), ("param", C.c_int32), ("expert", C.c_int32),
                ("row_block", C.c_int32), ("col_block", C.c_int32), ("ld", C.c_int32),
                ("rows_real", C.c_int16), ("cols_real", C.c_int16)]


class fp8z1_param_grid(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("first_block", "experts", "row_blocks", "col_blocks",
                                          "e_begin", "e_end")]


class fp8z1_adamw_hp(C.Structure):
    _fields_ = [("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float),
                ("eps", C.c_float), ("weight_decay", C.c_float), ("max_norm", C.c_float),
                ("loss_scale", C.c_float), ("step", C.c_int64)]


class fp8z1_step_scalars(C.Structure):
    _fields_ = [(n, C.c_float) for n in ("beta1", "beta2", "omb1", "omb2", "eps", "step_size",
                                          "inv_sqrt_bc2", "decay", "max_norm", "loss_scale")]


class fp8z1_loss_scaler(C.Structure):
    _fields_ = [("scale", C.c_float), ("step", C.c_int64), ("good_steps", C.c_int32),
                ("growth_interval", C.c_int32)]


BLOCK_DTYPE = np.dtype([("src_offset", "<i8"), ("param", "<i4"), ("expert", "<i4"),
                        ("row_block", "<i4"), ("col_block", "<i4"), ("ld", "<i4"),
                        ("rows_real", "<i2"), ("cols_real", "<i2")])
assert BLOCK_DTYPE.itemsize == C.sizeof(fp8z1_block) == 32

# every symbol the header declares, with (restype, argtypes)
_P = C.c_void_p
_SIGS = {
    "fp8z1_build_layout": (C.c_int, [C.POINTER(fp8z1_shape), C.c_int32, C.c_int32, C.c_uint32,
                                     C.POINTER(_P)]),
    "fp8z1_destroy_layout": (C.c_int, [_P]),
    "fp8z1_layout_info": (C.c_int, [_P, C.POINTER(C.c_int64), C.POINTER(C.c_int64),
                                    C.POINTER(C.c_int64)]),
    "fp8z1_shard_range": (C.c_int, [_P, C.c_int32, C.POINTER(C.c_int64), C.POINTER(C.c_int64)]),
    "fp8z1_copy_lut": (C.c_int, [_P, _P, C.c_int64]),
    "fp8z1_param_blocks": (C.c_int, [_P, C.c_int32, C.c_int64, C.c_int64, C.POINTER(fp8z1_param_grid)]),
    "fp8z1_device_status": (C.c_int, [_P, C.POINTER(C.c_uint32)]),
    "fp8z1_fold": (C.c_int, [_P, _P, _P, C.c_int32, C.c_int64, C.c_int64, _P]),
    "fp8z1_unfold": (C.c_int, [_P, _P, _P, C.c_int32, C.c_int64, C.c_int64, _P]),
    "fp8z1_grad_norm": (C.c_int, [_P, _P, C.c_int64, C.c_int64, _P, _P, _P]),
    "fp8z1_grad_norm_noalloc": (C.c_int, [_P, C.c_int64, _P, _P, _P]),
    "fp8z1_step": (C.c_int, [_P, C.POINTER(fp8z1_adamw_hp), _P, _P, _P, _P, _P, _P, C.c_int64,
                             C.c_int64, _P, _P, _P]),
    "fp8z1_fold_norm": (C.c_int, [_P, _P, _P, C.c_int64, C.c_int64, _P, _P, _P]),
    "fp8z1_step_fused": (C.c_int, [_P, C.POINTER(fp8z1_adamw_hp), _P, _P, _P, _P, _P, _P, _P, _P,
                                   _P, _P, C.c_int64, C.c_int64, _P, _P, _P]),
    "fp8z1_step_fused_dev": (C.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                       C.c_int64, C.c_int64, _P, _P, _P]),
    "fp8z1_step_fused_select": (C.c_int, [_P, C.POINTER(fp8z1_adamw_hp), C.POINTER(fp8z1_adamw_hp), _P, _P, _P,
                                          _P, _P, _P, _P, _P, _P, C.c_int64, C.c_int64, _P, _P, _P]),
    "fp8z1_graph_step_nodes": (C.c_int, [_P, _P, C.c_int32, C.POINTER(C.c_int32)]),
    "fp8z1_graph_set_step_hp": (C.c_int, [_P, _P, C.c_int32, C.POINTER(fp8z1_adamw_hp)]),
    "fp8z1_step_scalars_from_hp": (C.c_int, [C.POINTER(fp8z1_adamw_hp), C.POINTER(fp8z1_step_scalars)]),
    "fp8z1_paramwise_split": (C.c_int, [C.POINTER(fp8z1_shape), C.c_int32, C.c_int32, _P, _P,
                                        C.POINTER(C.c_int64)]),
    "fp8z1_mx_build_layout": (C.c_int, [C.POINTER(fp8z1_shape), C.c_int32, C.c_int32, C.c_uint32,
                                        C.POINTER(_P)]),
    "fp8z1_mx_destroy_layout": (C.c_int, [_P]),
    "fp8z1_mx_layout_info": (C.c_int, [_P, C.POINTER(C.c_int64), C.POINTER(C.c_int64)]),
    "fp8z1_mx_shard_range": (C.c_int, [_P, C.c_int32, C.POINTER(C.c_int64), C.POINTER(C.c_int64)]),
    "fp8z1_mx_grad_norm": (C.c_int, [_P, _P, C.c_int64, C.c_int64, _P, _P, _P]),
    "fp8z1_mx_step": (C.c_int, [_P, C.POINTER(fp8z1_adamw_hp), _P, _P, _P, _P, _P, _P, C.c_int64,
                                C.c_int64, _P, _P, _P]),
    "fp8z1_mx_step_select": (C.c_int, [_P, C.POINTER(fp8z1_adamw_hp), C.POINTER(fp8z1_adamw_hp), _P, _P, _P,
                                       _P, _P, _P, _P, C.c_int64, C.c_int64, _P, _P, _P]),
    "fp8z1_scaler_update": (C.c_int, [C.POINTER(fp8z1_loss_scaler), C.c_int32]),
    "fp8z1_clip_coef": (C.c_int, [C.c_double, C.c_float, C.c_float, C.POINTER(C.c_double),
                                  C.POINTER(C.c_double)]),
    "fp8z1_kernel_launches": (C.c_int, [C.POINTER(C.c_uint64)]),
    "fp8z1_build_flags": (C.c_int, []),
    "fp8z1_checked_misses": (C.c_int, [C.POINTER(C.c_uint64)]),
    "fp8z1_checked_set_lut_entry": (C.c_int, [_P, C.c_int64, _P]),
    "fp8z1_norm_reset": (C.c_int, [_P, _P, _P]),
    "fp8z1_strerror": (C.c_char_p, [C.c_int]),
}


def lib_path() -> str:
    return _LIB_PATH


def lib():
    """Load libfp8z1.so, or libfp8z1_checked.so under FP8Z1_CHECKED=1 (raises
    when it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(f"{os.path.basename(_LIB_PATH)} is not built ({_LIB_PATH}); "
                                   "run __graft_entry__.build()")
            L = C.CDLL(_LIB_PATH)
            for name, (res, args) in _SIGS.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(x)}")


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != OK:
        raise Fp8z1Error(status, where)


def fp8z1_strerror(status: int) -> str:
    return lib().fp8z1_strerror(int(status)).decode()


class Layout:
    """Owner of an ``fp8z1_layout*`` (freed with the object)."""

    def __init__(self, handle: int, shapes):
        self.handle = handle
        self.shapes = shapes

    def __del__(self):
        if getattr(self, "handle", None):
            try:
                lib().fp8z1_destroy_layout(self.handle)
            except Exception:
                pass
            self.handle = None

    @property
    def _as_parameter_(self):
        return self.handle


def _norm_shape(s):
    return (1, int(s[0]), int(s[1])) if len(s) == 2 else (int(s[0]), int(s[1]), int(s[2]))


def fp8z1_build_layout(shapes: Sequence[Sequence[int]], dp_size: int = 1,
                       host_only: bool = False) -> Layout:
    shapes = [_norm_shape(s) for s in shapes]
    arr = (fp8z1_shape * max(1, len(shapes)))(*[fp8z1_shape(*s) for s in shapes])
    out = _P()
    _check(lib().fp8z1_build_layout(arr, len(shapes), int(dp_size),
                                    LAYOUT_HOST_ONLY if host_only else 0, C.byref(out)),
           "fp8z1_build_layout")
    return Layout(out.value, shapes)


def fp8z1_layout_info(layout: Layout):
    a, b, c = C.c_int64(), C.c_int64(), C.c_int64()
    _check(lib().fp8z1_layout_info(layout.handle, C.byref(a), C.byref(b), C.byref(c)),
           "fp8z1_layout_info")
    return a.value, b.value, c.value


def fp8z1_shard_range(layout: Layout, rank: int):
    a, b = C.c_int64(), C.c_int64()
    _check(lib().fp8z1_shard_range(layout.handle, int(rank), C.byref(a), C.byref(b)),
           "fp8z1_shard_range")
    return a.value, b.value


def fp8z1_copy_lut(layout: Layout) -> np.ndarray:
    nblk = fp8z1_layout_info(layout)[0]
    out = np.zeros(max(1, nblk), dtype=BLOCK_DTYPE)
    _check(lib().fp8z1_copy_lut(layout.handle, out.ctypes.data, nblk), "fp8z1_copy_lut")
    return out[:nblk]


def fp8z1_param_blocks(layout: Layout, param: int, b0: int, b1: int) -> fp8z1_param_grid:
    """Where param ``param``'s blocks (and so its scales) sit in the flat
    block order, and the experts whose blocks all lie in [b0, b1)."""
    g = fp8z1_param_grid()
    _check(lib().fp8z1_param_blocks(layout.handle, int(param), int(b0), int(b1), C.byref(g)),
           "fp8z1_param_blocks")
    return g


def fp8z1_device_status(layout: Layout) -> int:
    v = C.c_uint32()
    _check(lib().fp8z1_device_status(layout.handle, C.byref(v)), "fp8z1_device_status")
    return v.value


def param_pointers(tensors, device=None):
    """Device int64 tensor holding the data pointers of ``tensors`` (the
    ``d_src_params`` / ``d_dst_params`` array of fold / unfold)."""
    import torch
    ptrs = [t.data_ptr() for t in tensors]
    dev = device if device is not None else tensors[0].device
    return torch.tensor(ptrs, dtype=torch.int64, device=dev)


def fp8z1_fold(layout: Layout, d_src_params, dst_shard, elem_size: int, b0: int, b1: int,
               stream=None):
    _check(lib().fp8z1_fold(layout.handle, _ptr(d_src_params), _ptr(dst_shard), int(elem_size),
                            int(b0), int(b1), _stream(stream)), "fp8z1_fold")


def fp8z1_unfold(layout: Layout, src_shard, d_dst_params, elem_size: int, b0: int, b1: int,
                 stream=None):
    _check(lib().fp8z1_unfold(layout.handle, _ptr(src_shard), _ptr(d_dst_params), int(elem_size),
                              int(b0), int(b1), _stream(stream)), "fp8z1_unfold")


def fp8z1_grad_norm(layout: Layout, grad_shard, b0: int, b1: int, d_sumsq, d_found_inf,
                    stream=None):
    _check(lib().fp8z1_grad_norm(layout.handle, _ptr(grad_shard), int(b0), int(b1), _ptr(d_sumsq),
                                 _ptr(d_found_inf), _stream(stream)), "fp8z1_grad_norm")


NOALLOC_MAX_BLOCKS = 262144


def fp8z1_grad_norm_noalloc(grad_shard, n_blocks: int, d_sumsq, d_found_inf, stream=None):
    """The grad norm of fp8z1_grad_norm for callers that cannot allocate
    device memory: no layout, a static device workspace, at most
    NOALLOC_MAX_BLOCKS blocks per call."""
    _check(lib().fp8z1_grad_norm_noalloc(_ptr(grad_shard), int(n_blocks), _ptr(d_sumsq),
                                         _ptr(d_found_inf), _stream(stream)),
           "fp8z1_grad_norm_noalloc")


def make_hp(lr, beta1, beta2, eps, weight_decay, max_norm, loss_scale, step) -> fp8z1_adamw_hp:
    return fp8z1_adamw_hp(lr, beta1, beta2, eps, weight_decay, max_norm, loss_scale, int(step))


def fp8z1_step(layout: Layout, hp: fp8z1_adamw_hp, grad_shard, master_shard, m_shard, v_shard,
               fp8_shard, scale_shard, b0: int, b1: int, d_sumsq, d_found_inf, stream=None):
    _check(lib().fp8z1_step(layout.handle, C.byref(hp), _ptr(grad_shard), _ptr(master_shard),
                            _ptr(m_shard), _ptr(v_shard), _ptr(fp8_shard), _ptr(scale_shard),
                            int(b0), int(b1), _ptr(d_sumsq), _ptr(d_found_inf), _stream(stream)),
           "fp8z1_step")


def fp8z1_fold_norm(layout: Layout, d_grad_params, grad_shard, b0: int, b1: int, d_sumsq,
                    d_found_inf, stream=None):
    """Fold (when grad_shard is not None) fused with the grad norm."""
    _check(lib().fp8z1_fold_norm(layout.handle, _ptr(d_grad_params), _ptr(grad_shard), int(b0),
                                 int(b1), _ptr(d_sumsq), _ptr(d_found_inf), _stream(stream)),
           "fp8z1_fold_norm")


def fp8z1_step_fused(layout: Layout, hp: fp8z1_adamw_hp, *, grad_shard=None, d_grad_params=None,
                     master_shard, m_shard, v_shard, fp8_shard=None, d_fp8_params=None,
                     scale_shard, block_cos=None, block_underflow=None, b0: int, b1: int, d_sumsq,
                     d_found_inf, stream=None):
    """fp8z1_step reading grads folded or row-major, writing codes folded
    and/or row-major, optionally with the per-block quantisation monitors."""
    _check(lib().fp8z1_step_fused(layout.handle, C.byref(hp), _ptr(grad_shard), _ptr(d_grad_params),
                                  _ptr(master_shard), _ptr(m_shard), _ptr(v_shard), _ptr(fp8_shard),
                                  _ptr(d_fp8_params), _ptr(scale_shard), _ptr(block_cos),
                                  _ptr(block_underflow), int(b0), int(b1),
                                  _ptr(d_sumsq), _ptr(d_found_inf), _stream(stream)),
           "fp8z1_step_fused")


def fp8z1_step_fused_dev(layout: Layout, h_scalars, d_scalars, *, grad_shard=None, d_grad_params=None,
                         master_shard, m_shard, v_shard, fp8_shard=None, d_fp8_params=None,
                         scale_shard, block_cos=None, block_underflow=None, b0: int, b1: int, d_sumsq,
                         d_found_inf, stream=None):
    """fp8z1_step_fused with the per-step scalars read from device memory
    ``d_scalars`` (40 bytes), after a copy from ``h_scalars`` (page-locked
    host memory, or None for no copy) enqueued on the same stream."""
    _check(lib().fp8z1_step_fused_dev(layout.handle, _ptr(h_scalars), _ptr(d_scalars), _ptr(grad_shard),
                                      _ptr(d_grad_params), _ptr(master_shard), _ptr(m_shard), _ptr(v_shard),
                                      _ptr(fp8_shard), _ptr(d_fp8_params), _ptr(scale_shard),
                                      _ptr(block_cos), _ptr(block_underflow), int(b0), int(b1),
                                      _ptr(d_sumsq), _ptr(d_found_inf), _stream(stream)),
           "fp8z1_step_fused_dev")


def fp8z1_step_fused_select(layout: Layout, hp_if_clear: fp8z1_adamw_hp, hp_if_set: fp8z1_adamw_hp,
                            d_select, *, grad_shard=None, d_grad_params=None, master_shard, m_shard, v_shard,
                            fp8_shard=None, d_fp8_params=None, scale_shard, b0: int, b1: int, d_sumsq,
                            d_found_inf, stream=None):
    """fp8z1_step_fused with ``hp_if_clear`` when *d_select == 0, else
    ``hp_if_set``, picked on the device when the kernel runs."""
    _check(lib().fp8z1_step_fused_select(layout.handle, C.byref(hp_if_clear), C.byref(hp_if_set), _ptr(d_select),
                                         _ptr(grad_shard), _ptr(d_grad_params), _ptr(master_shard), _ptr(m_shard),
                                         _ptr(v_shard), _ptr(fp8_shard), _ptr(d_fp8_params), _ptr(scale_shard),
                                         int(b0), int(b1), _ptr(d_sumsq), _ptr(d_found_inf), _stream(stream)),
           "fp8z1_step_fused_select")


def fp8z1_graph_step_nodes(graph: int):
    """The by-value step kernel nodes of a captured cudaGraph_t, as a ctypes
    array of node handles."""
    n = C.c_int32()
    st = lib().fp8z1_graph_step_nodes(C.c_void_p(graph), None, 0, C.byref(n))
    if st not in (OK, EINVAL) or (st == EINVAL and n.value == 0):
        _check(st, "fp8z1_graph_step_nodes")
    nodes = (C.c_void_p * max(1, n.value))()
    _check(lib().fp8z1_graph_step_nodes(C.c_void_p(graph), C.cast(nodes, C.c_void_p), n.value, C.byref(n)),
           "fp8z1_graph_step_nodes")
    return nodes, n.value


def fp8z1_graph_set_step_hp(graph_exec: int, nodes, n_nodes: int, hp: fp8z1_adamw_hp):
    """Rewrite the step scalars of those nodes in a cudaGraphExec_t."""
    _check(lib().fp8z1_graph_set_step_hp(C.c_void_p(graph_exec), C.cast(nodes, C.c_void_p), int(n_nodes),
                                         C.byref(hp)), "fp8z1_graph_set_step_hp")


def fp8z1_step_scalars_from_hp(hp: fp8z1_adamw_hp, out=None) -> fp8z1_step_scalars:
    """The FP32 scalars of one step (host).  ``out``: a tensor or address of
    40 bytes to fill in place (pinned host memory, say); the struct is
    returned either way."""
    sc = fp8z1_step_scalars()
    _check(lib().fp8z1_step_scalars_from_hp(C.byref(hp), C.byref(sc)), "fp8z1_step_scalars_from_hp")
    if out is not None:
        C.memmove(_ptr(out), C.addressof(sc), C.sizeof(sc))
    return sc


def fp8z1_norm_reset(d_sumsq, d_found_inf, stream=None):
    """*d_sumsq = 0, *d_found_inf = 0 (two memsets on ``stream``)."""
    _check(lib().fp8z1_norm_reset(_ptr(d_sumsq), _ptr(d_found_inf), _stream(stream)), "fp8z1_norm_reset")


def fp8z1_kernel_launches() -> int:
    """Kernels the library has enqueued in this process so far."""
    n = C.c_uint64()
    _check(lib().fp8z1_kernel_launches(C.byref(n)), "fp8z1_kernel_launches")
    return n.value


def fp8z1_build_flags() -> int:
    """BUILD_CHECKED for the checked library, else 0."""
    return int(lib().fp8z1_build_flags())


def fp8z1_checked_misses() -> int:
    """Row-major accesses the checked kernels skipped on the current device
    (synchronous; 0 in a release build)."""
    n = C.c_uint64()
    _check(lib().fp8z1_checked_misses(C.byref(n)), "fp8z1_checked_misses")
    return n.value


def fp8z1_checked_set_lut_entry(layout: Layout, block: int, entry: "fp8z1_block") -> None:
    """Checked builds' test hook: overwrite one device LUT entry."""
    _check(lib().fp8z1_checked_set_lut_entry(layout.handle, int(block), C.byref(entry)),
           "fp8z1_checked_set_lut_entry")


def fp8z1_paramwise_split(shapes, dp_size: int):
    """(owner[n], bucket_elems[dp], padded_total) of the greedy param-wise split."""
    shapes = [_norm_shape(s) for s in shapes]
    arr = (fp8z1_shape * max(1, len(shapes)))(*[fp8z1_shape(*s) for s in shapes])
    owner = np.zeros(max(1, len(shapes)), np.int32)
    bucket = np.zeros(max(1, dp_size), np.int64)
    padded = C.c_int64()
    _check(lib().fp8z1_paramwise_split(arr, len(shapes), int(dp_size), owner.ctypes.data,
                                       bucket.ctypes.data, C.byref(padded)), "fp8z1_paramwise_split")
    return owner[:len(shapes)], bucket[:dp_size], padded.value


class MxLayout(Layout):
    """Owner of an ``fp8z1_mx_layout*``."""

    def __del__(self):
        if getattr(self, "handle", None):
            try:
                lib().fp8z1_mx_destroy_layout(self.handle)
            except Exception:
                pass
            self.handle = None


def fp8z1_mx_build_layout(shapes, dp_size: int = 1, host_only: bool = False) -> MxLayout:
    shapes = [_norm_shape(s) for s in shapes]
    arr = (fp8z1_shape * max(1, len(shapes)))(*[fp8z1_shape(*s) for s in shapes])
    out = _P()
    _check(lib().fp8z1_mx_build_layout(arr, len(shapes), int(dp_size),
                                       LAYOUT_HOST_ONLY if host_only else 0, C.byref(out)),
           "fp8z1_mx_build_layout")
    return MxLayout(out.value, shapes)


def fp8z1_mx_layout_info(layout: MxLayout):
    a, b = C.c_int64(), C.c_int64()
    _check(lib().fp8z1_mx_layout_info(layout.handle, C.byref(a), C.byref(b)), "fp8z1_mx_layout_info")
    return a.value, b.value


def fp8z1_mx_shard_range(layout: MxLayout, rank: int):
    a, b = C.c_int64(), C.c_int64()
    _check(lib().fp8z1_mx_shard_range(layout.handle, int(rank), C.byref(a), C.byref(b)),
           "fp8z1_mx_shard_range")
    return a.value, b.value


def fp8z1_mx_grad_norm(layout: MxLayout, grad_shard, g0: int, g1: int, d_sumsq, d_found_inf,
                       stream=None):
    _check(lib().fp8z1_mx_grad_norm(layout.handle, _ptr(grad_shard), int(g0), int(g1), _ptr(d_sumsq),
                                    _ptr(d_found_inf), _stream(stream)), "fp8z1_mx_grad_norm")


def fp8z1_mx_step(layout: MxLayout, hp: fp8z1_adamw_hp, grad_shard, master_shard, m_shard, v_shard,
                  fp8_shard, scale_shard, g0: int, g1: int, d_sumsq, d_found_inf, stream=None):
    _check(lib().fp8z1_mx_step(layout.handle, C.byref(hp), _ptr(grad_shard), _ptr(master_shard),
                               _ptr(m_shard), _ptr(v_shard), _ptr(fp8_shard), _ptr(scale_shard),
                               int(g0), int(g1), _ptr(d_sumsq), _ptr(d_found_inf), _stream(stream)),
           "fp8z1_mx_step")


def fp8z1_mx_step_select(layout: MxLayout, hp_if_clear: fp8z1_adamw_hp, hp_if_set: fp8z1_adamw_hp, d_select,
                         grad_shard, master_shard, m_shard, v_shard, fp8_shard, scale_shard, g0: int, g1: int,
                         d_sumsq, d_found_inf, stream=None):
    """fp8z1_mx_step with ``hp_if_clear`` when *d_select == 0, else ``hp_if_set``."""
    _check(lib().fp8z1_mx_step_select(layout.handle, C.byref(hp_if_clear), C.byref(hp_if_set), _ptr(d_select),
                                      _ptr(grad_shard), _ptr(master_shard), _ptr(m_shard), _ptr(v_shard),
                                      _ptr(fp8_shard), _ptr(scale_shard), int(g0), int(g1), _ptr(d_sumsq),
                                      _ptr(d_found_inf), _stream(stream)), "fp8z1_mx_step_select")


def fp8z1_clip_coef(sumsq: float, max_norm: float, loss_scale: float):
    """(global_norm, clip_coef) of a step, as the device computes them."""
    g, c = C.c_double(), C.c_double()
    _check(lib().fp8z1_clip_coef(float(sumsq), float(max_norm), float(loss_scale), C.byref(g), C.byref(c)),
           "fp8z1_clip_coef")
    return g.value, c.value


def fp8z1_scaler_update(scaler: fp8z1_loss_scaler, found_inf: int):
    _check(lib().fp8z1_scaler_update(C.byref(scaler), int(found_inf)), "fp8z1_scaler_update")
