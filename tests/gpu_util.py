"""Helpers shared by the GPU parity tests: tolerances, dtype plumbing and
guarded output buffers. Expected values always come from the oracle."""
from __future__ import annotations

import numpy as np
import torch

import normalization_reduction_gb300 as fn

F32_TOL = 1e-4          # max-abs, fp32 outputs
BF16_TOL = 2e-2         # max-abs, bf16 outputs (or one bf16 ulp where larger)
CANARY = -12345.0


def dev() -> torch.device:
    return torch.device("cuda", torch.cuda.current_device())


def code(dtype) -> int:
    return fn.FNORM_F32 if dtype == torch.float32 else fn.FNORM_BF16


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 7), 2.0 ** -133)


def assert_close(got: np.ndarray, ref: np.ndarray, out_dtype, what: str = "") -> float:
    """|got - ref| within the output type's tolerance; returns the max error."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    if out_dtype == torch.bfloat16:
        tol = np.maximum(BF16_TOL, bf16_ulp(ref))
    else:
        tol = np.full(ref.shape, F32_TOL)
    bad = err > tol
    if np.any(bad):
        i = np.argmax(err - tol)
        raise AssertionError(f"{what}: {int(bad.sum())} of {err.size} outside tolerance; "
                             f"worst at flat {i}: got {got.flat[i]!r} ref {ref.flat[i]!r}")
    return float(err.max()) if err.size else 0.0


class Guarded:
    """A device buffer with canary bands in front of and behind the view."""

    def __init__(self, shape, dtype, band: int = 4096, offset_elems: int = 0):
        n = int(np.prod(shape)) if len(shape) else 1
        self.band = band + offset_elems
        self.buf = torch.full((n + 2 * band + offset_elems,), CANARY, dtype=dtype, device=dev())
        self.view = self.buf[self.band:self.band + n].view(shape)
        self.n = n

    def check(self):
        head = self.buf[:self.band]
        tail = self.buf[self.band + self.n:]
        assert bool((head == CANARY).all()), "write before the output buffer"
        assert bool((tail == CANARY).all()), "write past the output buffer"
