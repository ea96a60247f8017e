"""Helpers for the GPU parity tests (test infrastructure)."""
import numpy as np
import pytest
import torch

from blockwise_fp8_zero_fold_gb300 import build as fp8build
from blockwise_fp8_zero_fold_gb300 import fp8z1 as F

NP_OF = {4: np.float32, 2: np.uint16, 1: np.uint8}
TORCH_OF = {4: torch.float32, 2: torch.int16, 1: torch.uint8}


@pytest.fixture(scope="session")
def lib():
    fp8build.build(checked=F.CHECKED)
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return F.lib()


def to_host(t: torch.Tensor) -> np.ndarray:
    a = t.detach().cpu().numpy()
    return np.ascontiguousarray(a)


def bytes_of(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = to_host(a)
    return np.ascontiguousarray(a).view(np.uint8).reshape(-1)


def assert_rel(got: np.ndarray, want: np.ndarray, rtol: float, what: str):
    """|got - want| <= rtol*|want| elementwise; where want == 0, got == want."""
    got = got.astype(np.float64)
    want = want.astype(np.float64)
    bad = np.abs(got - want) > rtol * np.abs(want)
    if bad.any():
        i = np.flatnonzero(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements beyond rel {rtol}; "
                             f"first {i.tolist()}: got {got.reshape(-1)[i].tolist()} want {want.reshape(-1)[i].tolist()}")


def code_ordinal(q: np.ndarray) -> np.ndarray:
    """Signed ordinal of an E4M3 code (0x00 and 0x80 both map to 0)."""
    q = q.astype(np.int32)
    mag = q & 0x7F
    return np.where(q & 0x80, -mag, mag)


def assert_codes(got: np.ndarray, want: np.ndarray, what: str):
    """Within one code step everywhere, mismatching on at most 1e-4 of elements."""
    d = np.abs(code_ordinal(got) - code_ordinal(want))
    assert d.max(initial=0) <= 1, f"{what}: a code differs by {d.max()} steps"
    frac = float((d != 0).mean()) if d.size else 0.0
    assert frac <= 1e-4, f"{what}: {frac:.2e} of codes differ"
    return frac
