"""Affine InstanceNorm and eval-mode BatchNorm on the GPU through the C ABI
against the oracle: every InstanceNorm kernel shape with per-channel
gamma/beta (so that slice q must find channel q % C), each parameter alone,
vector and element-wise access, all dtype pairs; eval BatchNorm over short
runs (grid-stride kernel) and long runs (per-run kernel), ragged and
misaligned inputs, in place, guard bands, and running statistics produced by
a training call."""
import numpy as np
import pytest
import torch

import normalization_reduction_gb300 as fn
from normalization_reduction_gb300 import inputs
from tests.gpu_util import Guarded, assert_close, code, dev, to_f64

pytestmark = pytest.mark.gpu

EPS = 1e-5


def params(C, seed):
    g = torch.Generator().manual_seed(seed)
    gamma = (torch.randn(C, generator=g) * 0.7 + 1.0).to(dev())
    beta = (torch.randn(C, generator=g) * 0.5).to(dev())
    return gamma, beta


def run_affine(x, gamma, beta, N, C, S, out_dtype, out=None, stats=False):
    y = out if out is not None else torch.empty(x.shape, dtype=out_dtype, device=x.device)
    NC = N * C
    mean = torch.empty(max(NC, 1), device=x.device) if stats else None
    rstd = torch.empty(max(NC, 1), device=x.device) if stats else None
    fn.fnorm_instancenorm_affine(x, y, gamma, beta, N, C, S, code(x.dtype), code(out_dtype), EPS,
                                 mean, rstd)
    torch.cuda.synchronize()
    return y, mean, rstd


def oracle_affine(orc, x, gamma, beta, N, C, S):
    g = None if gamma is None else gamma.cpu().numpy()
    b = None if beta is None else beta.cpu().numpy()
    ref, mean, var = orc.instancenorm_affine(to_f64(x).reshape(N, C, S), g, b, EPS)
    return ref.reshape(x.shape), mean, var


def make_x(shape, dtype, seed):
    return inputs.normal(shape, seed, "cpu", mean=3.0, std=2.0).to(dtype).to(dev())


AFFINE_SIZES = [1, 7, 256, 1000, 4097, 16387, 65536, 262144]


@pytest.mark.parametrize("S", AFFINE_SIZES)
@pytest.mark.parametrize("dt", ["f32", "bf16", "bf16>f32", "f32>bf16"])
def test_affine_sizes_and_dtypes(orc, S, dt):
    tin = torch.bfloat16 if dt.startswith("bf16") else torch.float32
    tout = {"f32": torch.float32, "bf16": torch.bfloat16, "bf16>f32": torch.float32,
            "f32>bf16": torch.bfloat16}[dt]
    C = 5
    N = max(1, min(8, 1_500_000 // (S * C)))
    x = make_x((N, C, S), tin, 30_000 + S)
    gamma, beta = params(C, S)
    g = Guarded((N, C, S), tout)
    y, mean, rstd = run_affine(x, gamma, beta, N, C, S, tout, out=g.view, stats=True)
    g.check()
    ref, rmean, rvar = oracle_affine(orc, x, gamma, beta, N, C, S)
    assert_close(to_f64(y), ref, tout, f"affine S={S} {dt}")
    assert_close(mean.cpu().numpy()[:N * C], rmean, torch.float32, "mean")
    assert np.allclose(rstd.cpu().numpy()[:N * C], 1 / np.sqrt(rvar + EPS), rtol=2e-6, atol=0)


AFFINE_FORCED = [
    ("group:8:1", 20), ("group:32:4", 500), ("group:32:8", 1024),
    ("resident:256:8:1", 8000), ("resident:512:8:8", 100000),
    ("split:512:8:8:1", 32768), ("split:512:8:8:8", 200000), ("split:256:8:0:1", 4096),
    ("stream:1", 77777), ("stream:8", 262144),
]


@pytest.mark.parametrize("path,S", AFFINE_FORCED, ids=[p for p, _ in AFFINE_FORCED])
@pytest.mark.parametrize("scalar", [False, True], ids=["vec", "scalar"])
def test_affine_forced_paths(orc, fnorm_env, path, S, scalar):
    if path.startswith("split") and scalar:
        pytest.skip("the split kernel has vector access only")
    fnorm_env.setenv("FNORM_FORCE_PATH", path)
    if scalar:
        fnorm_env.setenv("FNORM_FORCE_SCALAR", "1")
    C = 3
    N = max(2, min(7, 2_000_000 // (S * C)))
    for tin in (torch.float32, torch.bfloat16):
        x = make_x((N, C, S), tin, 40_000 + S)
        gamma, beta = params(C, 7 + S)
        y, _, _ = run_affine(x, gamma, beta, N, C, S, tin)
        ref, _, _ = oracle_affine(orc, x, gamma, beta, N, C, S)
        assert_close(to_f64(y), ref, tin, f"{path} S={S} {tin}")


@pytest.mark.parametrize("which", ["gamma", "beta", "none"])
def test_affine_one_parameter(orc, which):
    N, C, S = 3, 4, 3000
    x = make_x((N, C, S), torch.float32, 51)
    gamma, beta = params(C, 52)
    gamma = gamma if which == "gamma" else None
    beta = beta if which == "beta" else None
    y, _, _ = run_affine(x, gamma, beta, N, C, S, torch.float32)
    ref, _, _ = oracle_affine(orc, x, gamma, beta, N, C, S)
    assert_close(to_f64(y), ref, torch.float32, which)
    if which == "none":
        y2 = torch.empty_like(x)
        fn.fnorm_instancenorm(x, y2, N, C, S, fn.FNORM_F32, fn.FNORM_F32, EPS, None, None)
        torch.cuda.synchronize()
        assert torch.equal(y, y2)


def test_affine_in_place_and_helper(orc):
    N, C, S = 4, 6, 4096
    x = make_x((N, C, 64, 64), torch.float32, 61)
    gamma, beta = params(C, 62)
    ref, _, _ = oracle_affine(orc, x, gamma, beta, N, C, S)
    y = fn.instance_norm(x, weight=gamma, bias=beta)
    assert_close(to_f64(y), ref, torch.float32, "helper")
    fn.fnorm_instancenorm_affine(x, x, gamma, beta, N, C, S, fn.FNORM_F32, fn.FNORM_F32, EPS,
                                 None, None)
    torch.cuda.synchronize()
    assert torch.equal(x, y)


# ---------------------------------------------------------------- eval BatchNorm
def run_eval(x, gamma, beta, scale, rm, rv, N, C, S, out=None):
    y = out if out is not None else torch.empty_like(x)
    fn.fnorm_batchnorm_eval(x, y, gamma, beta, scale, rm, rv, EPS, N, C, S)
    torch.cuda.synchronize()
    return y


def oracle_eval(orc, x, gamma, beta, scale, rm, rv, N, C, S):
    g = None if gamma is None else gamma.cpu().numpy()
    b = None if beta is None else beta.cpu().numpy()
    return orc.batchnorm_eval(to_f64(x).reshape(N, C, S), g, b, scale, rm.cpu().numpy(),
                              rv.cpu().numpy(), EPS)


EVAL_SHAPES = [(2, 3, 1), (4, 5, 7), (3, 4, 100), (2, 3, 1023), (2, 3, 1024), (5, 7, 4097),
               (3, 2, 16387), (8, 16, 15876), (1, 1, 40000), (64, 3, 3)]


@pytest.mark.parametrize("shape", EVAL_SHAPES, ids=[f"{n}x{c}x{s}" for n, c, s in EVAL_SHAPES])
@pytest.mark.parametrize("scalar", [False, True], ids=["vec", "scalar"])
@pytest.mark.parametrize("affine", [True, False], ids=["affine", "plain"])
@pytest.mark.parametrize("staged", ["1", "0"], ids=["staged", "registers"])
def test_eval_shapes(orc, fnorm_env, shape, scalar, affine, staged):
    if scalar:
        fnorm_env.setenv("FNORM_FORCE_SCALAR", "1")
    fnorm_env.setenv("FNORM_BN_SPLIT", staged)
    N, C, S = shape
    x, _, _ = inputs.per_channel_normal((N, C, S), 70_000 + S * C, dev())
    gamma, beta = params(C, 71 + S) if affine else (None, None)
    gr = torch.Generator().manual_seed(72 + S)
    rm = (torch.randn(C, generator=gr) * 0.3).to(dev())
    rv = (torch.rand(C, generator=gr) * 2.0 + 0.1).to(dev())
    g = Guarded((N, C, S), torch.float32)
    y = run_eval(x, gamma, beta, 2.0, rm, rv, N, C, S, out=g.view)
    g.check()
    ref = oracle_eval(orc, x, gamma, beta, 2.0, rm, rv, N, C, S)
    assert_close(to_f64(y), ref, torch.float32, f"eval {shape}")


@pytest.mark.parametrize("S", [1000, 15876])
def test_eval_misaligned_and_in_place(orc, S):
    """x and y one element past a 16-byte boundary take the element-wise path;
    in place (y == x) gives the same values."""
    N, C = 3, 4
    x0 = inputs.normal((N * C * S + 1,), 81, dev(), mean=0.2, std=1.5)
    x = x0[1:].view(N, C, S)
    gamma, beta = params(C, 82)
    rm = torch.linspace(-0.5, 0.5, C, device=dev())
    rv = torch.linspace(0.5, 2.0, C, device=dev())
    ref = oracle_eval(orc, x, gamma, beta, 2.0, rm, rv, N, C, S)
    yb = torch.empty(N * C * S + 1, device=dev())
    y = yb[1:].view(N, C, S)
    run_eval(x, gamma, beta, 2.0, rm, rv, N, C, S, out=y)
    assert_close(to_f64(y), ref, torch.float32, "misaligned")
    xc = x.contiguous().clone()
    run_eval(xc, gamma, beta, 2.0, rm, rv, N, C, S, out=xc)
    assert torch.equal(xc, run_eval(x.contiguous(), gamma, beta, 2.0, rm, rv, N, C, S))


def test_eval_after_training_call(orc):
    """Running statistics written by fnorm_batchnorm_train feed an eval call on
    the same stream; both match the oracle's train-then-eval sequence."""
    N, C, S = 16, 8, 900
    x, gamma, beta, rm, rv = inputs.batchnorm(dev(), (N, C, 30, 30), 91)
    rm0, rv0 = rm.cpu().numpy(), rv.cpu().numpy()
    y = torch.empty_like(x)
    ws = torch.empty(fn.fnorm_batchnorm_workspace_size(N, C, S), dtype=torch.uint8, device=dev())
    fn.fnorm_batchnorm_train(x, y, gamma, beta, 2.0, rm, rv, 0.1, EPS, None, None, N, C, S, ws,
                             ws.numel())
    x2, _, _ = inputs.per_channel_normal((N, C, 30, 30), 92, dev())
    y2 = fn.batch_norm_eval(x2, rm, rv, gamma, beta, eps=EPS, scale=2.0)
    torch.cuda.synchronize()
    _, rmo, rvo, _, _ = orc.batchnorm_train(x.cpu().numpy().reshape(N, C, S),
                                            gamma.cpu().numpy(), beta.cpu().numpy(), 2.0, rm0,
                                            rv0, 0.1, EPS)
    ref = orc.batchnorm_eval(to_f64(x2).reshape(N, C, S), gamma.cpu().numpy(),
                             beta.cpu().numpy(), 2.0, rmo, rvo, EPS)
    assert_close(to_f64(y2).reshape(N, C, S), ref, torch.float32, "train then eval")
