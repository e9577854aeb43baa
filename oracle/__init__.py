"""Oracle for libfnorm -- TEST INFRASTRUCTURE, NOT PRODUCT CODE.

A plain float64, single-threaded CPU statement of the library's operations
(``fnorm_oracle.cpp`` beside this file), wrapped with ctypes and numpy.
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it. It imports nothing from the CUDA package and the
CUDA package imports nothing from it.

Sources: the pages Kimi-K2.6__l2_p79 (the Conv3d -> InstanceNorm3d -> clamp ->
max epilogue), Kimi-K2.6__l2_p73 (Conv2d -> BatchNorm2d -> x2.0) and
Kimi-K2.6__l1_p34 (InstanceNorm2d(64)); each function cites its passage in
the C++ source.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(exact rationals, closed forms, library routines, invariants); none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "fnorm_oracle.cpp")
LIBRARY = os.path.join(_HERE, "libfnorm_oracle.so")
CXXFLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC"]

_lock = threading.Lock()

_f64p = ctypes.POINTER(ctypes.c_double)
_f32p = ctypes.POINTER(ctypes.c_float)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i64p = ctypes.POINTER(ctypes.c_int64)
_i64 = ctypes.c_int64
_f64 = ctypes.c_double


def compile_library(source: str = SOURCE, output: str = LIBRARY, extra_flags=()) -> str:
    """Compile ``source`` into the shared library ``output`` with g++ (atomic replace)."""
    out_dir = os.path.dirname(os.path.abspath(output))
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=out_dir)
    os.close(fd)
    try:
        cmd = ["g++", *CXXFLAGS, *extra_flags, source, "-o", tmp]
        subprocess.run(cmd, check=True, capture_output=True, text=True)
        os.replace(tmp, output)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return output


def build(force: bool = False) -> str:
    """Build ``libfnorm_oracle.so`` if it is missing or older than its source."""
    with _lock:
        stale = (not os.path.exists(LIBRARY)
                 or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE))
        if force or stale:
            compile_library()
    return LIBRARY


def _ptr(a: np.ndarray | None, typ):
    if a is None:
        return ctypes.cast(None, typ)
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(typ)


class Oracle:
    """ctypes view of one compiled oracle library (the real one by default)."""

    def __init__(self, path: str | None = None):
        self.path = path or build()
        lib = ctypes.CDLL(self.path)
        lib.fnorm_oracle_round_bf16.argtypes = [_f64p, _u16p, _i64]
        lib.fnorm_oracle_round_bf16.restype = None
        lib.fnorm_oracle_bf16_to_f64.argtypes = [_u16p, _f64p, _i64]
        lib.fnorm_oracle_bf16_to_f64.restype = None
        for name, xt, yt in (("fnorm_oracle_instancenorm_f64", _f64p, _f64p),
                             ("fnorm_oracle_instancenorm_f32", _f32p, _f32p),
                             ("fnorm_oracle_instancenorm_bf16", _u16p, _u16p)):
            fn = getattr(lib, name)
            fn.argtypes = [xt, yt, _i64, _i64, _f64, _f64p, _f64p]
            fn.restype = ctypes.c_int
        lib.fnorm_oracle_epilogue_f32.argtypes = [_f32p, _f32p, _f32p, _i64p, _f32p, _i64, _i64,
                                                  _i64, _f64, _f64, _f64]
        lib.fnorm_oracle_epilogue_f32.restype = ctypes.c_int
        lib.fnorm_oracle_batchnorm_train_f32.argtypes = [_f32p, _f32p, _f32p, _f32p, _f64, _f64p,
                                                         _f64p, _f64, _f64, _i64, _i64, _i64,
                                                         _f64p, _f64p]
        lib.fnorm_oracle_batchnorm_train_f32.restype = ctypes.c_int
        lib.fnorm_oracle_instancenorm_affine_f64.argtypes = [_f64p, _f64p, _f64p, _f64p, _i64,
                                                             _i64, _i64, _f64, _f64p, _f64p]
        lib.fnorm_oracle_instancenorm_affine_f64.restype = ctypes.c_int
        lib.fnorm_oracle_batchnorm_eval_f64.argtypes = [_f64p, _f64p, _f64p, _f64p, _f64, _f64p,
                                                        _f64p, _f64, _i64, _i64, _i64]
        lib.fnorm_oracle_batchnorm_eval_f64.restype = ctypes.c_int
        self.lib = lib

    # -- bf16 storage -----------------------------------------------------
    def round_bf16(self, v) -> np.ndarray:
        """float64 values -> nearest-even bf16 bit patterns (uint16)."""
        v = np.ascontiguousarray(v, dtype=np.float64)
        out = np.empty(v.shape, dtype=np.uint16)
        self.lib.fnorm_oracle_round_bf16(_ptr(v, _f64p), _ptr(out, _u16p), v.size)
        return out

    def bf16_to_f64(self, bits) -> np.ndarray:
        bits = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.empty(bits.shape, dtype=np.float64)
        self.lib.fnorm_oracle_bf16_to_f64(_ptr(bits, _u16p), _ptr(out, _f64p), bits.size)
        return out

    # -- InstanceNorm -----------------------------------------------------
    def instancenorm(self, x: np.ndarray, eps: float = 1e-5):
        """x [..., S] viewed as [NC, S] (float64, float32, or uint16 bf16 bits).

        Returns (y, mean, var): y has x's dtype and shape; mean/var are float64
        [NC] biased statistics.
        """
        x = np.ascontiguousarray(x)
        S = x.shape[-1] if x.ndim else 1
        NC = x.size // S if S else 0
        y = np.empty_like(x)
        mean = np.empty(NC, dtype=np.float64)
        var = np.empty(NC, dtype=np.float64)
        if x.dtype == np.float64:
            fn, t = self.lib.fnorm_oracle_instancenorm_f64, _f64p
        elif x.dtype == np.float32:
            fn, t = self.lib.fnorm_oracle_instancenorm_f32, _f32p
        elif x.dtype == np.uint16:
            fn, t = self.lib.fnorm_oracle_instancenorm_bf16, _u16p
        else:
            raise TypeError(f"unsupported dtype {x.dtype}")
        rc = fn(_ptr(x, t), _ptr(y, t), NC, S, float(eps), _ptr(mean, _f64p), _ptr(var, _f64p))
        if rc != 0:
            raise ValueError("oracle instancenorm rejected its arguments")
        return y, mean, var

    def instancenorm_affine(self, x: np.ndarray, gamma=None, beta=None, eps: float = 1e-5):
        """x [N, C, *spatial] (any real dtype, taken exactly in float64); gamma/beta
        [C] or None (1 / 0).

        Returns (y float64 of x's shape, mean [N*C], var [N*C]) in float64.
        """
        x = np.ascontiguousarray(x, dtype=np.float64)
        N, C = x.shape[0], x.shape[1]
        S = int(np.prod(x.shape[2:])) if x.ndim > 2 else 1
        g = None if gamma is None else np.ascontiguousarray(gamma, dtype=np.float64).reshape(-1)
        b = None if beta is None else np.ascontiguousarray(beta, dtype=np.float64).reshape(-1)
        y = np.empty_like(x)
        mean = np.empty(N * C, dtype=np.float64)
        var = np.empty(N * C, dtype=np.float64)
        rc = self.lib.fnorm_oracle_instancenorm_affine_f64(
            _ptr(x, _f64p), _ptr(y, _f64p), _ptr(g, _f64p), _ptr(b, _f64p), N, C, S, float(eps),
            _ptr(mean, _f64p), _ptr(var, _f64p))
        if rc != 0:
            raise ValueError("oracle instancenorm_affine rejected its arguments")
        return y, mean, var

    # -- fused epilogue ---------------------------------------------------
    def epilogue(self, x: np.ndarray, m: np.ndarray, eps: float = 1e-5, lo: float = -1.0,
                 hi: float = 1.0):
        """x [N, C, *spatial] float32, m [C] float32.

        Returns (y [N, *spatial] f32, argmax [N, *spatial] int64,
        second [N, *spatial] f32 runner-up value).
        """
        x = np.ascontiguousarray(x, dtype=np.float32)
        m = np.ascontiguousarray(m, dtype=np.float32).reshape(-1)
        N, C = x.shape[0], x.shape[1]
        spatial = x.shape[2:]
        S = int(np.prod(spatial)) if spatial else 1
        y = np.empty((N,) + spatial, dtype=np.float32)
        arg = np.empty((N,) + spatial, dtype=np.int64)
        second = np.empty((N,) + spatial, dtype=np.float32)
        rc = self.lib.fnorm_oracle_epilogue_f32(_ptr(x, _f32p), _ptr(m, _f32p), _ptr(y, _f32p),
                                                _ptr(arg, _i64p), _ptr(second, _f32p), N, C, S,
                                                float(eps), float(lo), float(hi))
        if rc != 0:
            raise ValueError("oracle epilogue rejected its arguments")
        return y, arg, second

    # -- BatchNorm (training) ---------------------------------------------
    def batchnorm_train(self, x: np.ndarray, gamma=None, beta=None, scale: float = 1.0,
                        running_mean=None, running_var=None, momentum: float = 0.1,
                        eps: float = 1e-5):
        """x [N, C, *spatial] float32; gamma/beta [C] float32 or None.

        Returns (y f32, new_running_mean f64 [C] or None, new_running_var f64 [C] or None,
        batch mean f64 [C], biased batch var f64 [C]).
        """
        x = np.ascontiguousarray(x, dtype=np.float32)
        N, C = x.shape[0], x.shape[1]
        S = int(np.prod(x.shape[2:])) if x.ndim > 2 else 1
        y = np.empty_like(x)
        g = None if gamma is None else np.ascontiguousarray(gamma, dtype=np.float32)
        b = None if beta is None else np.ascontiguousarray(beta, dtype=np.float32)
        rm = None if running_mean is None else np.array(running_mean, dtype=np.float64)
        rv = None if running_var is None else np.array(running_var, dtype=np.float64)
        mean = np.empty(C, dtype=np.float64)
        var = np.empty(C, dtype=np.float64)
        rc = self.lib.fnorm_oracle_batchnorm_train_f32(
            _ptr(x, _f32p), _ptr(y, _f32p), _ptr(g, _f32p), _ptr(b, _f32p), float(scale),
            _ptr(rm, _f64p), _ptr(rv, _f64p), float(momentum), float(eps), N, C, S,
            _ptr(mean, _f64p), _ptr(var, _f64p))
        if rc != 0:
            raise ValueError("oracle batchnorm rejected its arguments")
        return y, rm, rv, mean, var


    # -- BatchNorm (eval) -------------------------------------------------
    def batchnorm_eval(self, x: np.ndarray, gamma, beta, scale: float, running_mean,
                       running_var, eps: float = 1e-5) -> np.ndarray:
        """x [N, C, *spatial] (taken exactly in float64); gamma/beta [C] or None;
        running_mean/running_var [C]. Returns y float64 of x's shape."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        N, C = x.shape[0], x.shape[1]
        S = int(np.prod(x.shape[2:])) if x.ndim > 2 else 1
        g = None if gamma is None else np.ascontiguousarray(gamma, dtype=np.float64).reshape(-1)
        b = None if beta is None else np.ascontiguousarray(beta, dtype=np.float64).reshape(-1)
        rm = np.ascontiguousarray(running_mean, dtype=np.float64).reshape(-1)
        rv = np.ascontiguousarray(running_var, dtype=np.float64).reshape(-1)
        y = np.empty_like(x)
        rc = self.lib.fnorm_oracle_batchnorm_eval_f64(
            _ptr(x, _f64p), _ptr(y, _f64p), _ptr(g, _f64p), _ptr(b, _f64p), float(scale),
            _ptr(rm, _f64p), _ptr(rv, _f64p), float(eps), N, C, S)
        if rc != 0:
            raise ValueError("oracle batchnorm_eval rejected its arguments")
        return y


_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from ``fnorm_oracle.cpp`` (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
