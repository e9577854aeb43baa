"""The C ABI on the CPU: the library loads, exports every declared entry
point, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re
import subprocess

import pytest

import normalization_reduction_gb300 as fn
from normalization_reduction_gb300 import build as nbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "fnorm.h")


@pytest.fixture(scope="module")
def lib():
    nbuild.build()
    return fn.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fnorm_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("fnorm_instancenorm", "fnorm_instancenorm_epilogue",
                     "fnorm_batchnorm_train", "fnorm_batchnorm_workspace_size",
                     "fnorm_status_string", "fnorm_get_last_error", "fnorm_version"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_tuning_switches_read_once(lib, monkeypatch):
    """The FNORM_* switches are read once per process; fnorm_tuning_reload
    re-reads them, and the forced-timeout hook takes no environment input."""
    fn.fnorm_tuning_reload()
    monkeypatch.setenv("FNORM_DEBUG_FORCE_TIMEOUT", "1")   # no longer a switch
    fn.fnorm_tuning_reload()
    fn.fnorm_debug_force_timeout(False)
    monkeypatch.undo()
    fn.fnorm_tuning_reload()
    src = open(os.path.join(os.path.dirname(HEADER), "..", "normalization_reduction_gb300", "csrc",
                            "fnorm_api.cu")).read()
    assert "FNORM_DEBUG_FORCE_TIMEOUT" not in src
    assert src.count("std::getenv(") == 1   # only the one-time reader


def test_instancenorm_ws_validation(lib):
    """The workspace entry point validates like fnorm_instancenorm; its size is
    0 for shapes that do not take the workspace route."""
    assert fn.fnorm_instancenorm_workspace_size(112, 64, 512 * 512) == 0   # fits a cluster
    assert fn.fnorm_instancenorm_workspace_size(0, 1, 1 << 26) == 0
    assert fn.fnorm_instancenorm_workspace_size(1, 1, -1) == 0
    a = dict(x=FAKE, y=FAKE + (1 << 30), N=2, C=3, S=64, in_dtype=fn.FNORM_F32,
             out_dtype=fn.FNORM_F32, eps=1e-5, mean_out=None, rstd_out=None, workspace=None,
             workspace_bytes=0, stream=0)
    for kw, expect in [(dict(N=-1), fn.Status.ERR_INVALID_ARG),
                       (dict(eps=-1.0), fn.Status.ERR_INVALID_ARG),
                       (dict(x=FAKE + 2), fn.Status.ERR_ALIGNMENT),
                       (dict(N=0), fn.Status.OK)]:
        b = dict(a)
        b.update(kw)
        assert _rc(lambda: fn.fnorm_instancenorm_ws(**b)) == expect, kw


def test_injected_launch_failures(lib):
    """fnorm_debug_fail_launches(n): the next n calls that pass their checks
    return FNORM_ERR_CUDA before touching the GPU (fake pointers here); calls
    that fail their checks or are no-ops do not consume one."""
    a = dict(x=FAKE, y=FAKE + (1 << 30), N=2, C=3, S=64, in_dtype=fn.FNORM_F32,
             out_dtype=fn.FNORM_F32, eps=1e-5, mean_out=None, rstd_out=None, stream=0)
    fn.fnorm_debug_fail_launches(2)
    try:
        assert _rc(lambda: fn.fnorm_instancenorm(**dict(a, eps=-1.0))) == fn.Status.ERR_INVALID_ARG
        assert _rc(lambda: fn.fnorm_instancenorm(**dict(a, N=0))) == fn.Status.OK
        assert _rc(lambda: fn.fnorm_instancenorm(**a)) == fn.Status.ERR_CUDA
        assert _rc(lambda: fn.fnorm_instancenorm_epilogue(FAKE, FAKE + (1 << 31),
                                                          FAKE + (1 << 30), None, 2, 3, 64,
                                                          stream=0)) == fn.Status.ERR_CUDA
    finally:
        fn.fnorm_debug_fail_launches(0)


def test_status_strings_and_version(lib):
    for s in fn.Status:
        assert fn.fnorm_status_string(int(s)) == "FNORM_" + s.name
    assert fn.fnorm_version() >= 100


def _rc(call):
    try:
        call()
    except fn.FnormError as e:
        return e.status
    return fn.Status.OK


FAKE = 1 << 40   # never dereferenced: every case below fails validation first


@pytest.mark.parametrize("kw,expect", [
    (dict(N=-1), fn.Status.ERR_INVALID_ARG),
    (dict(eps=-1e-5), fn.Status.ERR_INVALID_ARG),
    (dict(eps=float("nan")), fn.Status.ERR_INVALID_ARG),
    (dict(eps=float("inf")), fn.Status.ERR_INVALID_ARG),
    (dict(in_dtype=7), fn.Status.ERR_INVALID_ARG),
    (dict(x=0), fn.Status.ERR_INVALID_ARG),
    (dict(x=FAKE + 2), fn.Status.ERR_ALIGNMENT),
    (dict(y=FAKE + 4, x=FAKE), fn.Status.ERR_INVALID_ARG),     # partial overlap
    (dict(y=FAKE, x=FAKE, out_dtype=fn.FNORM_BF16), fn.Status.ERR_INVALID_ARG),
    (dict(N=0), fn.Status.OK),                                  # empty: no-op
    (dict(S=0), fn.Status.OK),
    (dict(N=1 << 40, C=1 << 40), fn.Status.ERR_INVALID_ARG),   # size overflow
    (dict(mean_out=FAKE + 64, x=FAKE), fn.Status.ERR_INVALID_ARG),
])
def test_instancenorm_validation(lib, kw, expect):
    a = dict(x=FAKE, y=FAKE + (1 << 30), N=2, C=3, S=64, in_dtype=fn.FNORM_F32,
             out_dtype=fn.FNORM_F32, eps=1e-5, mean_out=None, rstd_out=None, stream=0)
    a.update(kw)
    assert _rc(lambda: fn.fnorm_instancenorm(**a)) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(C=0), fn.Status.ERR_INVALID_ARG),
    (dict(C=9000), fn.Status.ERR_UNSUPPORTED),
    (dict(clamp_lo=1.0, clamp_hi=-1.0), fn.Status.ERR_INVALID_ARG),
    (dict(clamp_lo=float("nan")), fn.Status.ERR_INVALID_ARG),
    (dict(m=0), fn.Status.ERR_INVALID_ARG),
    (dict(argmax=FAKE + (1 << 30) + 4), fn.Status.ERR_ALIGNMENT),
    (dict(y=FAKE + 128), fn.Status.ERR_INVALID_ARG),           # y inside x
    (dict(N=0), fn.Status.OK),
])
def test_epilogue_validation(lib, kw, expect):
    a = dict(x=FAKE, m=FAKE + (1 << 32), y=FAKE + (1 << 30), argmax=None, N=2, C=4, S=64,
             eps=1e-5, clamp_lo=-1.0, clamp_hi=1.0, stream=0)
    a.update(kw)
    assert _rc(lambda: fn.fnorm_instancenorm_epilogue(**a)) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(N=1, S=1), fn.Status.ERR_INVALID_ARG),                # needs two values per channel
    (dict(workspace_bytes=16), fn.Status.ERR_INVALID_ARG),
    (dict(workspace=FAKE + (1 << 34) + 16), fn.Status.ERR_ALIGNMENT),
    (dict(running_var=None), fn.Status.ERR_INVALID_ARG),       # both or neither
    (dict(momentum=float("nan")), fn.Status.ERR_INVALID_ARG),
    (dict(C=70000), fn.Status.ERR_UNSUPPORTED),
    (dict(workspace=FAKE + 256), fn.Status.ERR_INVALID_ARG),   # workspace inside x
    (dict(C=0), fn.Status.OK),
])
def test_batchnorm_validation(lib, kw, expect):
    a = dict(x=FAKE, y=FAKE + (1 << 30), gamma=None, beta=None, scale=2.0,
             running_mean=FAKE + (1 << 33), running_var=FAKE + (1 << 33) + 4096, momentum=0.1,
             eps=1e-5, save_mean=None, save_rstd=None, N=2, C=3, S=64,
             workspace=FAKE + (1 << 34), workspace_bytes=1 << 20, stream=0)
    a.update(kw)
    if "workspace_bytes" not in kw:
        a["workspace_bytes"] = max(fn.fnorm_batchnorm_workspace_size(a["N"], a["C"], a["S"]), 1 << 20)
    assert _rc(lambda: fn.fnorm_batchnorm_train(**a)) == expect


def test_workspace_size(lib):
    assert fn.fnorm_batchnorm_workspace_size(0, 4, 4) == 0
    w = fn.fnorm_batchnorm_workspace_size(128, 64, 126 * 126)
    assert w % 256 == 0 and w >= 64 * 128 * 16
    # one partial per (run, chunk of up to 16384 elements)
    assert fn.fnorm_batchnorm_workspace_size(2, 3, 40000) >= 3 * 2 * 3 * 16


@pytest.mark.parametrize("kw,expect", [
    (dict(R=0), fn.Status.ERR_INVALID_ARG),
    (dict(stats_all=FAKE + (1 << 35) + 4), fn.Status.ERR_ALIGNMENT),
    (dict(stats_all=0), fn.Status.ERR_INVALID_ARG),
    (dict(momentum=float("inf")), fn.Status.ERR_INVALID_ARG),
    (dict(N=0), fn.Status.OK),
])
def test_apply_stats_validation(lib, kw, expect):
    a = dict(x=FAKE, y=FAKE + (1 << 30), stats_all=FAKE + (1 << 35), R=2, gamma=None, beta=None,
             scale=1.0, running_mean=None, running_var=None, momentum=0.1, eps=1e-5,
             save_mean=None, save_rstd=None, N=2, C=3, S=64, stream=0)
    a.update(kw)
    assert _rc(lambda: fn.fnorm_batchnorm_apply_stats(**a)) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(stats_out=FAKE + (1 << 35) + 8), fn.Status.ERR_ALIGNMENT),
    (dict(workspace_bytes=16), fn.Status.ERR_INVALID_ARG),
    (dict(stats_out=FAKE + 64), fn.Status.ERR_INVALID_ARG),      # stats inside x
    (dict(C=0), fn.Status.OK),
])
def test_local_stats_validation(lib, kw, expect):
    a = dict(x=FAKE, stats_out=FAKE + (1 << 35), N=2, C=3, S=64, workspace=FAKE + (1 << 34),
             workspace_bytes=1 << 20, stream=0)
    a.update(kw)
    assert _rc(lambda: fn.fnorm_batchnorm_local_stats(**a)) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(gamma=FAKE + (1 << 36) + 2), fn.Status.ERR_ALIGNMENT),
    (dict(beta=FAKE + (1 << 36) + 1), fn.Status.ERR_ALIGNMENT),
    (dict(gamma=FAKE + (1 << 30) + 8), fn.Status.ERR_INVALID_ARG),   # gamma inside y
    (dict(beta=FAKE + (1 << 30)), fn.Status.ERR_INVALID_ARG),        # beta inside y
    (dict(eps=-1.0), fn.Status.ERR_INVALID_ARG),
    (dict(N=0), fn.Status.OK),
])
def test_instancenorm_affine_validation(lib, kw, expect):
    a = dict(x=FAKE, y=FAKE + (1 << 30), gamma=FAKE + (1 << 36), beta=FAKE + (1 << 36) + 4096,
             N=2, C=3, S=64, in_dtype=fn.FNORM_F32, out_dtype=fn.FNORM_F32, eps=1e-5,
             mean_out=None, rstd_out=None, stream=0)
    a.update(kw)
    assert _rc(lambda: fn.fnorm_instancenorm_affine(**a)) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(running_mean=None), fn.Status.ERR_INVALID_ARG),         # running statistics required
    (dict(running_var=None), fn.Status.ERR_INVALID_ARG),
    (dict(running_var=FAKE + (1 << 33) + 4098), fn.Status.ERR_ALIGNMENT),
    (dict(y=None), fn.Status.ERR_INVALID_ARG),
    (dict(y=FAKE + 4), fn.Status.ERR_INVALID_ARG),                # partial overlap with x
    (dict(running_mean=FAKE + 64), fn.Status.ERR_INVALID_ARG),    # statistics inside x
    (dict(scale=float("nan")), fn.Status.ERR_INVALID_ARG),
    (dict(eps=float("inf")), fn.Status.ERR_INVALID_ARG),
    (dict(C=70000), fn.Status.ERR_UNSUPPORTED),
    (dict(N=0), fn.Status.OK),
    (dict(S=0), fn.Status.OK),
])
def test_batchnorm_eval_validation(lib, kw, expect):
    a = dict(x=FAKE, y=FAKE + (1 << 30), gamma=None, beta=None, scale=2.0,
             running_mean=FAKE + (1 << 33), running_var=FAKE + (1 << 33) + 4096, eps=1e-5,
             N=2, C=3, S=64, stream=0)
    a.update(kw)
    assert _rc(lambda: fn.fnorm_batchnorm_eval(**a)) == expect


C_CALLER = r"""
#include <stdio.h>
#include "fnorm.h"
int call_all(void* x, void* y, float* g, float* m, long long* a, void* ws, fnorm_stream_t s) {
  fnorm_status st = fnorm_instancenorm(x, y, 2, 3, 64, FNORM_F32, FNORM_BF16, 1e-5f, 0, 0, s);
  st = fnorm_instancenorm_affine(x, y, g, g, 2, 3, 64, FNORM_BF16, FNORM_F32, 1e-5f, 0, 0, s);
  st = fnorm_instancenorm_epilogue((const float*)x, m, (float*)y, (int64_t*)a, 2, 3, 64, 1e-5f,
                                   -1.f, 1.f, s);
  size_t wb = fnorm_batchnorm_workspace_size(2, 3, 64);
  st = fnorm_batchnorm_train((const float*)x, (float*)y, g, g, 2.f, g, g, 0.1f, 1e-5f, 0, 0,
                             2, 3, 64, ws, wb, s);
  st = fnorm_batchnorm_eval((const float*)x, (float*)y, g, g, 2.f, g, g, 1e-5f, 2, 3, 64, s);
  st = fnorm_batchnorm_local_stats((const float*)x, g, 2, 3, 64, ws, wb, s);
  st = fnorm_batchnorm_apply_stats((const float*)x, (float*)y, g, 1, g, g, 2.f, g, g, 0.1f,
                                   1e-5f, 0, 0, 2, 3, 64, s);
  st = fnorm_batchnorm_train_noalloc((const float*)x, (float*)y, g, g, 2.f, g, g, 0.1f, 1e-5f,
                                     0, 0, 2, 3, 64, s);
  size_t iw = fnorm_instancenorm_workspace_size(1, 1, 1 << 26);
  st = fnorm_instancenorm_ws(x, y, 2, 3, 64, FNORM_F32, FNORM_F32, 1e-5f, 0, 0, ws, iw, s);
  fnorm_tuning_reload();
  fnorm_debug_force_timeout(0);
  fnorm_debug_fail_launches(0);
  printf("%s %d %d\n", fnorm_status_string(st), (int)fnorm_get_last_error(), fnorm_version());
  return (int)st;
}
"""


def test_header_is_plain_c(tmp_path, lib):
    """A C caller of every entry point compiles against include/fnorm.h with
    gcc (no CUDA headers) and links against libfnorm.so."""
    src = tmp_path / "caller.c"
    src.write_text(C_CALLER)
    inc = os.path.dirname(HEADER)
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", inc, "-c", str(src), "-o",
                        str(tmp_path / "caller.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    so = tmp_path / "libcaller.so"
    r = subprocess.run(["gcc", "-shared", str(tmp_path / "caller.o"), "-o", str(so),
                        fn.LIBRARY, "-Wl,--no-undefined", "-Wl,--allow-shlib-undefined"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
