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


def check_in_chunks(n_units: int, chunk: int, fetch, check, workers: int | None = None) -> int:
    """Runs ``check(a, b, fetch(a, b))`` for every chunk [a, b) of ``n_units``.

    ``fetch`` (device -> host copies) runs in the calling thread, ``check``
    (the oracle and the comparison) in a pool of threads: the oracle's ctypes
    calls and numpy's array arithmetic release the GIL, so chunks are checked
    in parallel on the host cores while the next chunk is copied. At most
    ``2 * workers`` fetched chunks are held at once. Returns the number of
    chunks checked; any failing check raises here.
    """
    import concurrent.futures as cf
    import os

    workers = workers or max(1, min(8, (os.cpu_count() or 2) - 1))
    done = 0
    with cf.ThreadPoolExecutor(max_workers=workers) as pool:
        pending = []
        for a in range(0, n_units, chunk):
            b = min(n_units, a + chunk)
            host = fetch(a, b)
            pending.append(pool.submit(check, a, b, host))
            while len(pending) >= 2 * workers:
                pending.pop(0).result()
                done += 1
        for f in pending:
            f.result()
            done += 1
    return done


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16 or int16) -> float64, exactly."""
    u = np.ascontiguousarray(bits).view(np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def host_bits(t: torch.Tensor) -> np.ndarray:
    """A bf16 device tensor's bit patterns on the host (uint16)."""
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)
