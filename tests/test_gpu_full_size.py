"""Parity at the benchmark's full sizes, element by element on every slice,
sample or channel, in the launch configuration bench.py times (the library's
default plan). Expected values come from the oracle, run chunk by chunk on the
host cores (tests/gpu_util.check_in_chunks):

* InstanceNorm fp32 x[112,64,512,512] (InstanceNorm2d(64), page
  Kimi-K2.6__l1_p34, block 1): all 7168 slices, and every slice's mean and
  rstd outputs; the output moments (mean 0, biased variance var/(var+eps)) are
  checked as well, as an extra.
* Epilogue fp32 x[128,16,14,30,30] (page Kimi-K2.6__l2_p79, block 1): the
  whole output, with the argmax output (argmax bit-exact where the oracle's
  top two differ) and without it (the saturating-clamp kernel that the
  benchmark times).
* BatchNorm fp32 x[128,64,126,126] (page Kimi-K2.6__l2_p73, block 1): the
  whole output, running statistics and saved statistics.
* bf16 sweep, 2^30 elements for each slice length S = 4^4 ... 4^10: every
  slice.
* Affine InstanceNorm fp32 x[112,64,512,512]: every slice.
* Eval BatchNorm fp32 x[128,64,126,126]: every sample.
* InstanceNorm fp32 x[132,64,512,512] (more than 2^31 elements): every slice.
* fnorm_instancenorm_ws on x[1,1,8192,8192] (one slice of 67 M values).
* fnorm_instancenorm_ws on x[1,1,8192,8192] (one slice of 67 M values).
* Counts above 2^24 that are not powers of two (the statistics carry fp32
  counts): InstanceNorm slices of 4097 x 4097 and 4096 x 4100 values, and
  BatchNorm channels of 3 * 2^23 + 5 and 3 * (2^23 + 4) values, on the
  element-wise and the vector paths.
"""
import numpy as np
import pytest
import torch

import normalization_reduction_gb300 as fn
from normalization_reduction_gb300 import inputs
from tests.gpu_util import assert_close, bf16_bits_to_f64, check_in_chunks, dev, host_bits

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

EPS = 1e-5


def check_instancenorm_all_slices(orc, xv, yv, mean=None, rstd=None, what="", chunk=128):
    """Every slice of xv/yv ([NC, S] fp32 device views) against the oracle;
    mean/rstd ([NC] device) too when given."""
    NC = xv.shape[0]
    mean_h = mean.cpu().numpy() if mean is not None else None
    rstd_h = rstd.cpu().numpy() if rstd is not None else None

    def fetch(a, b):
        return xv[a:b].cpu().numpy(), yv[a:b].cpu().numpy()

    def check(a, b, host):
        xs, ys = host
        ref, rmean, rvar = orc.instancenorm(xs, EPS)
        assert_close(ys, ref, torch.float32, f"{what} slices {a}..{b - 1}")
        if mean_h is not None:
            assert_close(mean_h[a:b], rmean, torch.float32, f"{what} mean {a}..{b - 1}")
        if rstd_h is not None:
            assert np.allclose(rstd_h[a:b], 1 / np.sqrt(rvar + EPS), rtol=2e-6, atol=0), what

    assert check_in_chunks(NC, chunk, fetch, check) == -(-NC // chunk)


def test_instancenorm_large_full_size(orc):
    N, C, H, W = inputs.SHAPE_LARGE
    NC, S = N * C, H * W
    x = inputs.instancenorm_large(dev())
    y = torch.empty_like(x)
    mean = torch.empty(NC, device=dev())
    rstd = torch.empty(NC, device=dev())
    fn.fnorm_instancenorm(x, y, N, C, S, fn.FNORM_F32, fn.FNORM_F32, EPS, mean, rstd)
    torch.cuda.synchronize()
    xv, yv = x.view(NC, S), y.view(NC, S)
    check_instancenorm_all_slices(orc, xv, yv, mean, rstd, "C2")
    # extra: every slice's output mean ~ 0 and output variance ~ var/(var+eps)
    ym = yv.double().mean(dim=1)
    yvar = yv.double().var(dim=1, unbiased=False)
    xvar = xv.double().var(dim=1, unbiased=False)
    assert float(ym.abs().max()) < 1e-5
    assert float((yvar - xvar / (xvar + EPS)).abs().max()) < 1e-5


@pytest.mark.parametrize("want_arg", [True, False], ids=["argmax", "values_only"])
def test_epilogue_full_size(orc, want_arg):
    """The whole [128,14,30,30] output; without the argmax output this is the
    launch the benchmark times (all 128 samples' clusters, saturating clamp)."""
    x, m = inputs.epilogue(dev())
    N, C = x.shape[0], x.shape[1]
    S = x[0, 0].numel()
    y = torch.empty((N, S), device=dev())
    arg = torch.empty((N, S), dtype=torch.int64, device=dev()) if want_arg else None
    fn.fnorm_instancenorm_epilogue(x, m, y, arg, N, C, S, EPS, -1.0, 1.0)
    torch.cuda.synchronize()
    assert fn.fnorm_get_last_error() == fn.Status.OK
    ref, rarg, second = orc.epilogue(x.cpu().numpy().reshape(N, C, S), m.cpu().numpy(), EPS)
    assert_close(y.cpu().numpy(), ref, torch.float32, "C3")
    if want_arg:
        clear = (ref - second) > 1e-5
        assert clear.mean() > 0.99
        assert np.array_equal(arg.cpu().numpy()[clear], rarg[clear])


def test_batchnorm_full_size(orc):
    x, g, b, rm, rv = inputs.batchnorm(dev())
    N, C = x.shape[0], x.shape[1]
    S = x[0, 0].numel()
    rm0, rv0 = rm.cpu().numpy(), rv.cpu().numpy()
    y = torch.empty_like(x)
    ws = torch.empty(fn.fnorm_batchnorm_workspace_size(N, C, S), dtype=torch.uint8, device=dev())
    sm, sr = torch.empty(C, device=dev()), torch.empty(C, device=dev())
    fn.fnorm_batchnorm_train(x, y, g, b, 2.0, rm, rv, 0.1, EPS, sm, sr, N, C, S, ws, ws.numel())
    torch.cuda.synchronize()
    ref, rmo, rvo, mean, var = orc.batchnorm_train(x.cpu().numpy().reshape(N, C, S),
                                                   g.cpu().numpy(), b.cpu().numpy(), 2.0,
                                                   rm0, rv0, 0.1, EPS)
    assert_close(y.cpu().numpy().reshape(N, C, S), ref, torch.float32, "C4")
    assert np.max(np.abs(rm.cpu().numpy() - rmo)) <= 1e-6
    assert np.max(np.abs(rv.cpu().numpy() - rvo)) <= 2e-6
    assert np.max(np.abs(sm.cpu().numpy() - mean)) <= 1e-5
    assert np.allclose(sr.cpu().numpy(), 1 / np.sqrt(var + EPS), rtol=2e-6, atol=0)


@pytest.mark.parametrize("S", inputs.SWEEP_S)
def test_sweep_full_size(orc, S):
    """Every slice of the 2^30-element bf16 input (bf16 in, bf16 out)."""
    x = inputs.instancenorm_sweep(S, dev())
    N, C, _ = x.shape
    y = torch.empty_like(x)
    fn.fnorm_instancenorm(x, y, N, C, S, fn.FNORM_BF16, fn.FNORM_BF16, EPS, None, None)
    torch.cuda.synchronize()
    NC = N * C
    xv, yv = x.view(NC, S), y.view(NC, S)
    chunk = max(1, (1 << 25) // S)   # 32 Mi elements per chunk

    def fetch(a, b):
        return host_bits(xv[a:b]), host_bits(yv[a:b])

    def check(a, b, host):
        xb, yb = host
        ref_bits, _, _ = orc.instancenorm(xb, EPS)
        assert_close(bf16_bits_to_f64(yb), bf16_bits_to_f64(ref_bits), torch.bfloat16,
                     f"C5 S={S} slices {a}..{b - 1}")

    check_in_chunks(NC, chunk, fetch, check)
    del x, y
    torch.cuda.empty_cache()


def test_instancenorm_affine_full_size(orc):
    """Affine InstanceNorm fp32 x[112,64,512,512] with per-channel gamma/beta:
    every slice against the oracle, two samples (128 slices) per chunk."""
    x, gamma, beta = inputs.instancenorm_affine(dev())
    N, C, H, W = x.shape
    S = H * W
    y = torch.empty_like(x)
    fn.fnorm_instancenorm_affine(x, y, gamma, beta, N, C, S, fn.FNORM_F32, fn.FNORM_F32, EPS,
                                 None, None)
    torch.cuda.synchronize()
    g, b = gamma.cpu().numpy(), beta.cpu().numpy()
    xv, yv = x.view(N, C, S), y.view(N, C, S)

    def fetch(a, c):
        return xv[a:c].cpu().numpy(), yv[a:c].cpu().numpy()

    def check(a, c, host):
        xs, ys = host
        ref, _, _ = orc.instancenorm_affine(xs, g, b, EPS)
        assert_close(ys, ref, torch.float32, f"affine samples {a}..{c - 1}")

    check_in_chunks(N, 2, fetch, check)
    del x, y
    torch.cuda.empty_cache()


def test_batchnorm_eval_full_size(orc):
    """Eval BatchNorm fp32 x[128,64,126,126] with running statistics: every
    sample against the oracle."""
    x, g, b, rm, rv = inputs.batchnorm_eval(dev())
    N, C = x.shape[0], x.shape[1]
    S = x[0, 0].numel()
    y = torch.empty_like(x)
    fn.fnorm_batchnorm_eval(x, y, g, b, 2.0, rm, rv, EPS, N, C, S)
    torch.cuda.synchronize()
    gh, bh, rmh, rvh = (t.cpu().numpy() for t in (g, b, rm, rv))
    xv, yv = x.view(N, C, S), y.view(N, C, S)

    def fetch(a, c):
        return xv[a:c].cpu().numpy(), yv[a:c].cpu().numpy()

    def check(a, c, host):
        xs, ys = host
        ref = orc.batchnorm_eval(xs, gh, bh, 2.0, rmh, rvh, EPS)
        assert_close(ys, ref, torch.float32, f"eval BN samples {a}..{c - 1}")

    check_in_chunks(N, 8, fetch, check)


def test_instancenorm_beyond_2e31_elements(orc):
    """x[132,64,512,512] fp32 = 2.21e9 elements (> 2^31; 8.9 GB each way):
    every slice, including those around the element offsets 2^30 (byte offset
    2^32) and 2^31."""
    shape = (132, 64, 512, 512)
    N, C, H, W = shape
    NC, S = N * C, H * W
    assert NC * S > 2 ** 31
    x = inputs.instancenorm_large(dev(), shape=shape, seed=1102)
    y = torch.empty_like(x)
    fn.fnorm_instancenorm(x, y, N, C, S, fn.FNORM_F32, fn.FNORM_F32, EPS, None, None)
    torch.cuda.synchronize()
    check_instancenorm_all_slices(orc, x.view(NC, S), y.view(NC, S), what="> 2^31")
    del x, y
    torch.cuda.empty_cache()


@pytest.mark.parametrize("S", [4097 * 4097, 4096 * 4100], ids=["odd", "vector"])
def test_instancenorm_count_above_2e24(orc, S):
    """One slice of more than 2^24 values that is not a power of two: 4097 x
    4097 = 16,785,409 (element-wise paths) and 4096 x 4100 = 16,793,600
    (16-byte vector paths). The merged fp32 counts round; the result must
    still match the oracle."""
    assert S > 2 ** 24 and S & (S - 1) != 0
    for dtype in (torch.float32, torch.bfloat16):
        x = inputs.normal((1, 1, S), 1201, dev(), mean=3.0, std=2.0, dtype=dtype)
        y = torch.empty_like(x)
        mean = torch.empty(1, device=dev())
        rstd = torch.empty(1, device=dev())
        code = fn.FNORM_F32 if dtype == torch.float32 else fn.FNORM_BF16
        fn.fnorm_instancenorm(x, y, 1, 1, S, code, code, EPS, mean, rstd)
        torch.cuda.synchronize()
        if dtype == torch.float32:
            ref, rmean, rvar = orc.instancenorm(x.cpu().numpy().reshape(1, S), EPS)
            assert_close(y.cpu().numpy().reshape(1, S), ref, torch.float32, "S > 2^24 f32")
        else:
            ref_bits, rmean, rvar = orc.instancenorm(host_bits(x).reshape(1, S), EPS)
            assert_close(bf16_bits_to_f64(host_bits(y)).reshape(1, S),
                         bf16_bits_to_f64(ref_bits), torch.bfloat16, "S > 2^24 bf16")
        assert abs(float(mean.item()) - rmean[0]) <= 1e-5
        assert abs(float(rstd.item()) * np.sqrt(rvar[0] + EPS) - 1) <= 2e-6


@pytest.mark.parametrize("N,S", [(7, 3595119), (3, 8388612)], ids=["odd", "vector"])
def test_batchnorm_count_above_2e24(orc, N, S):
    """BatchNorm with more than 2^24 values per channel, not a power of two,
    over 2 channels: 7 x 3,595,119 = 3 * 2^23 + 5 (element-wise path) and
    3 x 8,388,612 = 25,165,836 (16-byte vector path)."""
    C = 2
    assert N * S > 2 ** 24 and (N * S) & (N * S - 1) != 0
    x, _, _ = inputs.per_channel_normal((N, C, S), 1202, dev())
    g, b = inputs.channel_affine(C, 1202, dev())
    rm = torch.zeros(C, device=dev())
    rv = torch.ones(C, device=dev())
    y = torch.empty_like(x)
    ws = torch.empty(fn.fnorm_batchnorm_workspace_size(N, C, S), dtype=torch.uint8, device=dev())
    sm, sr = torch.empty(C, device=dev()), torch.empty(C, device=dev())
    fn.fnorm_batchnorm_train(x, y, g, b, 2.0, rm, rv, 0.1, EPS, sm, sr, N, C, S, ws, ws.numel())
    torch.cuda.synchronize()
    ref, rmo, rvo, mean, var = orc.batchnorm_train(x.cpu().numpy(), g.cpu().numpy(),
                                                   b.cpu().numpy(), 2.0, np.zeros(C),
                                                   np.ones(C), 0.1, EPS)
    assert_close(y.cpu().numpy(), ref, torch.float32, "BN count > 2^24")
    assert np.max(np.abs(rm.cpu().numpy() - rmo)) <= 1e-6
    assert np.max(np.abs(rv.cpu().numpy() - rvo)) <= 2e-6
    assert np.max(np.abs(sm.cpu().numpy() - mean)) <= 1e-5
    assert np.allclose(sr.cpu().numpy(), 1 / np.sqrt(var + EPS), rtol=2e-6, atol=0)


def test_instancenorm_workspace_route_largest_slice(orc):
    """fnorm_instancenorm_ws on x[1,1,8192,8192] fp32 (one slice of 67 M
    values: the chunked statistics, the per-slice merge launch and the apply
    pass), every element and the mean/rstd outputs against the oracle."""
    N, C, S = 1, 1, 8192 * 8192
    x = inputs.normal((N, C, S), 1401, dev(), mean=0.25, std=3.0)
    y = torch.empty_like(x)
    mean = torch.empty(1, device=dev())
    rstd = torch.empty(1, device=dev())
    nb = fn.fnorm_instancenorm_workspace_size(N, C, S)
    assert nb > 0
    ws = torch.empty(nb, dtype=torch.uint8, device=dev())
    fn.fnorm_instancenorm_ws(x, y, N, C, S, fn.FNORM_F32, fn.FNORM_F32, EPS, mean, rstd, ws, nb)
    torch.cuda.synchronize()
    check_instancenorm_all_slices(orc, x.view(1, S), y.view(1, S), mean, rstd, "ws 8192^2",
                                  chunk=1)
    del x, y
    torch.cuda.empty_cache()
