"""Python binding of libfnorm (include/fnorm.h): argument marshalling only.

The functions named ``fnorm_*`` mirror the C ABI one to one: they take device
pointers (ints) or CUDA tensors (their ``data_ptr()`` is passed), shapes and a
stream (``None`` = torch's current stream, a ``torch.cuda.Stream`` or a raw
handle), call the shared library and raise :class:`FnormError` on a non-OK
status. Every step of the computation runs in the library's CUDA kernels;
there is no fallback of any kind -- when ``libfnorm.so`` is missing the
functions raise.

The lower-case helpers at the end (``instance_norm``, ``instance_norm_epilogue``,
``batch_norm_train``) allocate outputs with torch and call the same entry
points.
"""
from __future__ import annotations

import ctypes
import os
from enum import IntEnum

__all__ = [
    "FNORM_F32", "FNORM_BF16", "Status", "FnormError", "LIBRARY", "lib",
    "fnorm_instancenorm", "fnorm_instancenorm_affine", "fnorm_instancenorm_epilogue",
    "fnorm_instancenorm_workspace_size", "fnorm_instancenorm_ws",
    "fnorm_batchnorm_workspace_size", "fnorm_batchnorm_eval",
    "fnorm_batchnorm_train", "fnorm_batchnorm_train_noalloc", "fnorm_batchnorm_local_stats",
    "fnorm_batchnorm_apply_stats", "fnorm_status_string", "fnorm_get_last_error", "fnorm_version",
    "fnorm_tuning_reload", "fnorm_debug_force_timeout", "fnorm_debug_fail_launches",
    "instance_norm", "instance_norm_epilogue", "batch_norm_train", "batch_norm_eval",
]

LIBRARY = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfnorm.so")

FNORM_F32 = 0
FNORM_BF16 = 1


class Status(IntEnum):
    OK = 0
    ERR_INVALID_ARG = 1
    ERR_UNSUPPORTED = 2
    ERR_ALIGNMENT = 3
    ERR_CUDA = 4
    ERR_TIMEOUT = 5


class FnormError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = Status(status)
        super().__init__(f"{where}: {self.status.name}")


_lib = None
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_f32 = ctypes.c_float
_int = ctypes.c_int

# name -> (argtypes, restype)
_SIGNATURES = {
    "fnorm_instancenorm": ([_vp, _vp, _i64, _i64, _i64, _int, _int, _f32, _vp, _vp, _vp], _int),
    "fnorm_instancenorm_affine": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _f32, _vp,
                                   _vp, _vp], _int),
    "fnorm_instancenorm_workspace_size": ([_i64, _i64, _i64], ctypes.c_size_t),
    "fnorm_instancenorm_ws": ([_vp, _vp, _i64, _i64, _i64, _int, _int, _f32, _vp, _vp, _vp,
                               ctypes.c_size_t, _vp], _int),
    "fnorm_batchnorm_eval": ([_vp, _vp, _vp, _vp, _f32, _vp, _vp, _f32, _i64, _i64, _i64, _vp],
                             _int),
    "fnorm_instancenorm_epilogue": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _f32, _f32, _f32, _vp],
                                    _int),
    "fnorm_batchnorm_workspace_size": ([_i64, _i64, _i64], ctypes.c_size_t),
    "fnorm_batchnorm_train": ([_vp, _vp, _vp, _vp, _f32, _vp, _vp, _f32, _f32, _vp, _vp, _i64,
                               _i64, _i64, _vp, ctypes.c_size_t, _vp], _int),
    "fnorm_batchnorm_train_noalloc": ([_vp, _vp, _vp, _vp, _f32, _vp, _vp, _f32, _f32, _vp, _vp,
                                       _i64, _i64, _i64, _vp], _int),
    "fnorm_batchnorm_local_stats": ([_vp, _vp, _i64, _i64, _i64, _vp, ctypes.c_size_t, _vp], _int),
    "fnorm_batchnorm_apply_stats": ([_vp, _vp, _vp, _i64, _vp, _vp, _f32, _vp, _vp, _f32, _f32, _vp,
                                     _vp, _i64, _i64, _i64, _vp], _int),
    "fnorm_status_string": ([_int], ctypes.c_char_p),
    "fnorm_get_last_error": ([], _int),
    "fnorm_version": ([], _int),
    "fnorm_tuning_reload": ([], None),
    "fnorm_debug_force_timeout": ([_int], None),
    "fnorm_debug_fail_launches": ([_int], None),
}


def lib() -> ctypes.CDLL:
    """The loaded libfnorm.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIBRARY):
            raise RuntimeError(
                f"{LIBRARY} is missing: build it with `python -m normalization_reduction_gb300.build` "
                "(the library has no CPU or PyTorch fallback)")
        handle = ctypes.CDLL(LIBRARY)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.argtypes = args
            fn.restype = res
        _lib = handle
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if isinstance(s, int):
        return s
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return s.cuda_stream


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise FnormError(rc, where)


# ---------------------------------------------------------------- C ABI mirror
def fnorm_instancenorm(x, y, N, C, S, in_dtype, out_dtype, eps=1e-5, mean_out=None,
                       rstd_out=None, stream=None) -> None:
    _check(lib().fnorm_instancenorm(_ptr(x), _ptr(y), N, C, S, in_dtype, out_dtype, eps,
                                    _ptr(mean_out), _ptr(rstd_out), _stream(stream)),
           "fnorm_instancenorm")


def fnorm_instancenorm_affine(x, y, gamma, beta, N, C, S, in_dtype, out_dtype, eps=1e-5,
                              mean_out=None, rstd_out=None, stream=None) -> None:
    _check(lib().fnorm_instancenorm_affine(_ptr(x), _ptr(y), _ptr(gamma), _ptr(beta), N, C, S,
                                           in_dtype, out_dtype, eps, _ptr(mean_out),
                                           _ptr(rstd_out), _stream(stream)),
           "fnorm_instancenorm_affine")


def fnorm_instancenorm_workspace_size(N, C, S) -> int:
    return int(lib().fnorm_instancenorm_workspace_size(N, C, S))


def fnorm_instancenorm_ws(x, y, N, C, S, in_dtype, out_dtype, eps, mean_out, rstd_out, workspace,
                          workspace_bytes, stream=None):
    _check(lib().fnorm_instancenorm_ws(_ptr(x), _ptr(y), N, C, S, in_dtype, out_dtype, eps,
                                       _ptr(mean_out), _ptr(rstd_out), _ptr(workspace),
                                       workspace_bytes, _stream(stream)),
           "fnorm_instancenorm_ws")


def fnorm_instancenorm_epilogue(x, m, y, argmax, N, C, S, eps=1e-5, clamp_lo=-1.0, clamp_hi=1.0,
                                stream=None) -> None:
    _check(lib().fnorm_instancenorm_epilogue(_ptr(x), _ptr(m), _ptr(y), _ptr(argmax), N, C, S,
                                             eps, clamp_lo, clamp_hi, _stream(stream)),
           "fnorm_instancenorm_epilogue")


def fnorm_batchnorm_workspace_size(N, C, S) -> int:
    return int(lib().fnorm_batchnorm_workspace_size(N, C, S))


def fnorm_batchnorm_eval(x, y, gamma, beta, scale, running_mean, running_var, eps, N, C, S,
                         stream=None) -> None:
    _check(lib().fnorm_batchnorm_eval(_ptr(x), _ptr(y), _ptr(gamma), _ptr(beta), scale,
                                      _ptr(running_mean), _ptr(running_var), eps, N, C, S,
                                      _stream(stream)),
           "fnorm_batchnorm_eval")


def fnorm_batchnorm_train(x, y, gamma, beta, scale, running_mean, running_var, momentum, eps,
                          save_mean, save_rstd, N, C, S, workspace, workspace_bytes,
                          stream=None) -> None:
    _check(lib().fnorm_batchnorm_train(_ptr(x), _ptr(y), _ptr(gamma), _ptr(beta), scale,
                                       _ptr(running_mean), _ptr(running_var), momentum, eps,
                                       _ptr(save_mean), _ptr(save_rstd), N, C, S,
                                       _ptr(workspace), workspace_bytes, _stream(stream)),
           "fnorm_batchnorm_train")


def fnorm_batchnorm_train_noalloc(x, y, gamma, beta, scale, running_mean, running_var, momentum,
                                  eps, save_mean, save_rstd, N, C, S, stream=None) -> None:
    """fnorm_batchnorm_train for callers that cannot allocate: the library's
    own 2 MiB device scratch stands in for the workspace (see include/fnorm.h)."""
    _check(lib().fnorm_batchnorm_train_noalloc(_ptr(x), _ptr(y), _ptr(gamma), _ptr(beta), scale,
                                               _ptr(running_mean), _ptr(running_var), momentum,
                                               eps, _ptr(save_mean), _ptr(save_rstd), N, C, S,
                                               _stream(stream)),
           "fnorm_batchnorm_train_noalloc")


def fnorm_batchnorm_local_stats(x, stats_out, N, C, S, workspace, workspace_bytes,
                                stream=None) -> None:
    _check(lib().fnorm_batchnorm_local_stats(_ptr(x), _ptr(stats_out), N, C, S, _ptr(workspace),
                                             workspace_bytes, _stream(stream)),
           "fnorm_batchnorm_local_stats")


def fnorm_batchnorm_apply_stats(x, y, stats_all, R, gamma, beta, scale, running_mean, running_var,
                                momentum, eps, save_mean, save_rstd, N, C, S, stream=None) -> None:
    _check(lib().fnorm_batchnorm_apply_stats(_ptr(x), _ptr(y), _ptr(stats_all), R, _ptr(gamma),
                                             _ptr(beta), scale, _ptr(running_mean),
                                             _ptr(running_var), momentum, eps, _ptr(save_mean),
                                             _ptr(save_rstd), N, C, S, _stream(stream)),
           "fnorm_batchnorm_apply_stats")


def fnorm_status_string(status: int) -> str:
    return lib().fnorm_status_string(int(status)).decode()


def fnorm_get_last_error() -> Status:
    return Status(lib().fnorm_get_last_error())


def fnorm_version() -> int:
    return int(lib().fnorm_version())


def fnorm_tuning_reload() -> None:
    """Re-reads the FNORM_* tuning switches from the environment (tests and
    experiments; the library reads them once per process otherwise)."""
    lib().fnorm_tuning_reload()


def fnorm_debug_fail_launches(n: int) -> None:
    """Test hook: the next n computing calls that pass their argument checks
    return FNORM_ERR_CUDA without launching; 0 clears it."""
    lib().fnorm_debug_fail_launches(int(n))


def fnorm_debug_force_timeout(on: bool) -> None:
    """Test hook: later launches with a bounded-wait hook make one CTA's wait
    expire (FNORM_ERR_TIMEOUT in the error word); False turns it off."""
    lib().fnorm_debug_force_timeout(1 if on else 0)


# ---------------------------------------------------------------- torch helpers
def _dtype_code(dtype) -> int:
    import torch
    if dtype == torch.float32:
        return FNORM_F32
    if dtype == torch.bfloat16:
        return FNORM_BF16
    raise TypeError(f"unsupported dtype {dtype}")


def _need_cuda_contig(t, name):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def instance_norm(x, eps: float = 1e-5, out_dtype=None, out=None, return_stats: bool = False,
                  stream=None, weight=None, bias=None):
    """InstanceNorm of x [N, C, *spatial] over the spatial dims; with
    ``weight``/``bias`` ([C] fp32 CUDA tensors) the affine form
    y = xhat * weight[c] + bias[c]."""
    import torch
    _need_cuda_contig(x, "x")
    N, C = x.shape[0], x.shape[1]
    S = 1
    for d in x.shape[2:]:
        S *= d
    y = out if out is not None else torch.empty(x.shape, dtype=out_dtype or x.dtype,
                                                 device=x.device)
    mean = rstd = None
    if return_stats:
        mean = torch.empty(N * C, dtype=torch.float32, device=x.device)
        rstd = torch.empty(N * C, dtype=torch.float32, device=x.device)
    if weight is None and bias is None and y.data_ptr() == x.data_ptr():
        # in place, few slices too long for one cluster need a workspace to
        # use every SM (out of place the library keeps their statistics in y)
        nb = fnorm_instancenorm_workspace_size(N, C, S)
        ws = torch.empty(nb, dtype=torch.uint8, device=x.device) if nb else None
        fnorm_instancenorm_ws(x, y, N, C, S, _dtype_code(x.dtype), _dtype_code(y.dtype), eps,
                              mean, rstd, ws, nb, stream)
    elif weight is None and bias is None:
        fnorm_instancenorm(x, y, N, C, S, _dtype_code(x.dtype), _dtype_code(y.dtype), eps, mean,
                           rstd, stream)
    else:
        fnorm_instancenorm_affine(x, y, weight, bias, N, C, S, _dtype_code(x.dtype),
                                  _dtype_code(y.dtype), eps, mean, rstd, stream)
    return (y, mean, rstd) if return_stats else y


def instance_norm_epilogue(x, m, eps: float = 1e-5, clamp_lo: float = -1.0,
                           clamp_hi: float = 1.0, return_argmax: bool = False, stream=None):
    """max_c m_c * clamp(InstanceNorm(x * m_c), lo, hi) for x [N, C, *spatial] fp32."""
    import torch
    _need_cuda_contig(x, "x")
    _need_cuda_contig(m, "m")
    N, C = x.shape[0], x.shape[1]
    S = 1
    for d in x.shape[2:]:
        S *= d
    y = torch.empty((N,) + tuple(x.shape[2:]), dtype=torch.float32, device=x.device)
    arg = torch.empty(y.shape, dtype=torch.int64, device=x.device) if return_argmax else None
    fnorm_instancenorm_epilogue(x, m, y, arg, N, C, S, eps, clamp_lo, clamp_hi, stream)
    return (y, arg) if return_argmax else y


def batch_norm_train(x, gamma=None, beta=None, running_mean=None, running_var=None,
                     momentum: float = 0.1, eps: float = 1e-5, scale: float = 1.0,
                     workspace=None, out=None, return_stats: bool = False, stream=None):
    """Training-mode BatchNorm of x [N, C, *spatial] fp32, times ``scale``;
    updates running_mean/running_var in place when given."""
    import torch
    _need_cuda_contig(x, "x")
    N, C = x.shape[0], x.shape[1]
    S = 1
    for d in x.shape[2:]:
        S *= d
    y = out if out is not None else torch.empty_like(x)
    nbytes = fnorm_batchnorm_workspace_size(N, C, S)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=x.device)
    save_mean = save_rstd = None
    if return_stats:
        save_mean = torch.empty(C, dtype=torch.float32, device=x.device)
        save_rstd = torch.empty(C, dtype=torch.float32, device=x.device)
    fnorm_batchnorm_train(x, y, gamma, beta, scale, running_mean, running_var, momentum, eps,
                          save_mean, save_rstd, N, C, S, workspace, workspace.numel(), stream)
    return (y, save_mean, save_rstd) if return_stats else y


def batch_norm_eval(x, running_mean, running_var, gamma=None, beta=None, eps: float = 1e-5,
                    scale: float = 1.0, out=None, stream=None):
    """Eval-mode BatchNorm of x [N, C, *spatial] fp32 with the running
    statistics, times ``scale``; nothing is updated."""
    import torch
    _need_cuda_contig(x, "x")
    N, C = x.shape[0], x.shape[1]
    S = 1
    for d in x.shape[2:]:
        S *= d
    y = out if out is not None else torch.empty_like(x)
    fnorm_batchnorm_eval(x, y, gamma, beta, scale, running_mean, running_var, eps, N, C, S, stream)
    return y
