"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times (the library's default plan):

* InstanceNorm fp32 x[112,64,512,512]: 64 sampled slices (first, last and
  seeded random ones) against the oracle, plus, for every slice, the
  properties any correct output has (mean 0, biased variance var/(var+eps)).
* Epilogue fp32 x[128,16,14,30,30]: the whole output and argmax against the
  oracle.
* BatchNorm fp32 x[128,64,126,126]: the whole output, running statistics and
  saved statistics against the oracle.
* bf16 sweep, 2^30 elements for each slice length S = 4^4 ... 4^10: 16
  sampled slices per S against the oracle.
* Affine InstanceNorm fp32 x[112,64,512,512]: 16 sampled slices.
* Eval BatchNorm fp32 x[128,64,126,126]: five sampled samples n.
* InstanceNorm fp32 x[132,64,512,512] (more than 2^31 elements): slices around the 32-bit
  element and byte boundaries.
"""
import numpy as np
import pytest
import torch

import normalization_reduction_gb300 as fn
from normalization_reduction_gb300 import inputs
from tests.gpu_util import assert_close, dev, to_f64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

EPS = 1e-5


def sample_slices(NC, k, seed):
    rng = np.random.default_rng(seed)
    pick = set([0, 1, NC - 2, NC - 1]) | set(rng.choice(NC, size=k - 4, replace=False).tolist())
    return np.array(sorted(pick))


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
    idx = sample_slices(NC, 64, 7)
    ti = torch.from_numpy(idx).to(dev())
    xs = xv.index_select(0, ti).cpu().numpy()
    ref, rmean, rvar = orc.instancenorm(xs, EPS)
    assert_close(yv.index_select(0, ti).cpu().numpy(), ref, torch.float32, "C2 sampled")
    assert_close(mean[ti].cpu().numpy(), rmean, torch.float32, "C2 mean")
    assert np.allclose(rstd[ti].cpu().numpy(), 1 / np.sqrt(rvar + EPS), rtol=2e-6, atol=0)
    # every slice: output mean ~ 0 and output variance ~ var/(var+eps) ~ 1
    ym = yv.double().mean(dim=1)
    yvar = yv.double().var(dim=1, unbiased=False)
    xvar = xv.double().var(dim=1, unbiased=False)
    assert float(ym.abs().max()) < 1e-5
    assert float((yvar - xvar / (xvar + EPS)).abs().max()) < 1e-5


def test_epilogue_full_size(orc):
    x, m = inputs.epilogue(dev())
    N, C = x.shape[0], x.shape[1]
    S = x[0, 0].numel()
    y = torch.empty((N, S), device=dev())
    arg = torch.empty((N, S), dtype=torch.int64, device=dev())
    fn.fnorm_instancenorm_epilogue(x, m, y, arg, N, C, S, EPS, -1.0, 1.0)
    torch.cuda.synchronize()
    ref, rarg, second = orc.epilogue(x.cpu().numpy().reshape(N, C, S), m.cpu().numpy(), EPS)
    assert_close(y.cpu().numpy(), ref, torch.float32, "C3")
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
    x = inputs.instancenorm_sweep(S, dev())
    N, C, _ = x.shape
    y = torch.empty_like(x)
    fn.fnorm_instancenorm(x, y, N, C, S, fn.FNORM_BF16, fn.FNORM_BF16, EPS, None, None)
    torch.cuda.synchronize()
    NC = N * C
    idx = torch.from_numpy(sample_slices(NC, 16, S)).to(dev())
    xs = x.view(NC, S).index_select(0, idx)
    ys = y.view(NC, S).index_select(0, idx)
    ref, _, _ = orc.instancenorm(to_f64(xs), EPS)
    assert_close(to_f64(ys), ref, torch.bfloat16, f"C5 S={S}")
    del x, y
    torch.cuda.empty_cache()


def test_instancenorm_affine_full_size(orc):
    """Affine InstanceNorm fp32 x[112,64,512,512] with per-channel gamma/beta:
    16 sampled slices against the oracle (channel q % 64 for slice q)."""
    x, gamma, beta = inputs.instancenorm_affine(dev())
    N, C, H, W = x.shape
    NC, S = N * C, H * W
    y = torch.empty_like(x)
    fn.fnorm_instancenorm_affine(x, y, gamma, beta, N, C, S, fn.FNORM_F32, fn.FNORM_F32, EPS,
                                 None, None)
    torch.cuda.synchronize()
    idx = sample_slices(NC, 16, 11)
    ti = torch.from_numpy(idx).to(dev())
    xs = x.view(NC, S).index_select(0, ti).cpu().numpy().astype(np.float64)
    ys = y.view(NC, S).index_select(0, ti).cpu().numpy()
    g, b = gamma.cpu().numpy(), beta.cpu().numpy()
    for row, q in enumerate(idx):
        c = int(q) % C
        ref, _, _ = orc.instancenorm_affine(xs[row].reshape(1, 1, S), g[c:c + 1], b[c:c + 1], EPS)
        assert_close(ys[row], ref.reshape(S), torch.float32, f"affine slice {q}")
    del x, y
    torch.cuda.empty_cache()


def test_batchnorm_eval_full_size(orc):
    """Eval BatchNorm fp32 x[128,64,126,126] with running statistics: samples
    n = 0, 1, 63, 126, 127 against the oracle, whole output finite."""
    x, g, b, rm, rv = inputs.batchnorm_eval(dev())
    N, C = x.shape[0], x.shape[1]
    S = x[0, 0].numel()
    y = torch.empty_like(x)
    fn.fnorm_batchnorm_eval(x, y, g, b, 2.0, rm, rv, EPS, N, C, S)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(y).all())
    pick = torch.tensor([0, 1, 63, 126, 127], device=dev())
    xs = x.index_select(0, pick).cpu().numpy().reshape(5, C, S)
    ref = orc.batchnorm_eval(xs, g.cpu().numpy(), b.cpu().numpy(), 2.0, rm.cpu().numpy(),
                             rv.cpu().numpy(), EPS)
    assert_close(y.index_select(0, pick).cpu().numpy().reshape(5, C, S), ref, torch.float32,
                 "eval BN")


def test_instancenorm_beyond_2e31_elements(orc):
    """x[132,64,512,512] fp32 = 2.21e9 elements (> 2^31; 8.9 GB each way): slices around the
    element offsets 2^30 (byte offset 2^32) and 2^31, and the last slices, against the oracle."""
    shape = (132, 64, 512, 512)
    N, C, H, W = shape
    NC, S = N * C, H * W
    assert NC * S > 2 ** 31
    x = inputs.instancenorm_large(dev(), shape=shape, seed=1102)
    y = torch.empty_like(x)
    fn.fnorm_instancenorm(x, y, N, C, S, fn.FNORM_F32, fn.FNORM_F32, EPS, None, None)
    torch.cuda.synchronize()
    idx = np.array([0, 4095, 4096, 4097, 8191, 8192, 8193, NC - 2, NC - 1])
    ti = torch.from_numpy(idx).to(dev())
    xs = x.view(NC, S).index_select(0, ti).cpu().numpy()
    ref, _, _ = orc.instancenorm(xs, EPS)
    assert_close(y.view(NC, S).index_select(0, ti).cpu().numpy(), ref, torch.float32, "> 2^31")
    del x, y
    torch.cuda.empty_cache()
