"""Seeded random cases for every entry point against the oracle: random
shapes across the size classes of each kernel family, dtype pairs, affine
parameters present or not, misaligned (element-aligned) pointers, in-place
calls and guard bands. Each case is drawn from its own seed, so a failure
names a reproducible case."""
import numpy as np
import pytest
import torch

import normalization_reduction_gb300 as fn
from normalization_reduction_gb300 import inputs
from tests.gpu_util import Guarded, assert_close, code, dev, to_f64

pytestmark = pytest.mark.gpu

EPS = 1e-5
CASES = 40


def _slice_len(rng):
    # log-uniform over 1 .. 2^21, with a bias to multiples of the vector width
    S = int(np.exp(rng.uniform(0.0, np.log(2 ** 21))))
    if rng.random() < 0.6:
        S = max(8, S - S % 8)
    return S


def _offset_view(n, dtype, misalign, fill=None):
    buf = torch.empty(n + 1, dtype=dtype, device=dev())
    if fill is not None:
        buf.copy_(fill)
    return buf[1:] if misalign else buf[:n]


@pytest.mark.parametrize("case", range(CASES))
def test_fuzz_instancenorm(orc, case):
    rng = np.random.default_rng(9000 + case)
    S = _slice_len(rng)
    C = int(rng.integers(1, 9))
    N = int(max(1, min(6, 3_000_000 // (S * C))))
    tin = torch.bfloat16 if rng.random() < 0.4 else torch.float32
    tout = torch.bfloat16 if rng.random() < 0.3 else torch.float32
    misalign = rng.random() < 0.2
    affine = rng.random() < 0.5
    x = inputs.normal((N * C * S + 1,), 9100 + case, dev(), mean=float(rng.uniform(-3, 3)),
                      std=float(rng.uniform(0.1, 4.0))).to(tin)
    xv = x[1:] if misalign else x[:N * C * S]
    g = Guarded((N * C * S,), tout)
    gamma = beta = None
    if affine:
        gamma, beta = inputs.channel_affine(C, 9200 + case, dev())
    fn.fnorm_instancenorm_affine(xv, g.view, gamma, beta, N, C, S, code(tin), code(tout), EPS,
                                 None, None)
    torch.cuda.synchronize()
    g.check()
    ref, _, _ = orc.instancenorm_affine(to_f64(xv).reshape(N, C, S),
                                        None if gamma is None else gamma.cpu().numpy(),
                                        None if beta is None else beta.cpu().numpy(), EPS)
    assert_close(to_f64(g.view).reshape(N, C, S), ref, tout,
                 f"case {case}: N={N} C={C} S={S} {tin}->{tout} misalign={misalign}")


@pytest.mark.parametrize("case", range(20))
def test_fuzz_bf16_one_cta_slices(orc, case):
    """bf16 slices of 2049-4096 values: one 64-thread CTA per slice, statistics
    in one pass of shifted sums and packed pairs; slice lengths that fill the
    threads' slots or leave some empty, both output types, offset and spread
    drawn per case."""
    rng = np.random.default_rng(9700 + case)
    S = int(rng.integers(2049, 4097))
    if rng.random() < 0.6:
        S -= S % 8
    C, N = int(rng.integers(1, 9)), int(rng.integers(1, 40))
    tout = torch.bfloat16 if rng.random() < 0.5 else torch.float32
    x = inputs.normal((N * C * S,), 9800 + case, dev(), mean=float(rng.uniform(-5, 5)),
                      std=float(rng.uniform(0.05, 4.0))).to(torch.bfloat16)
    g = Guarded((N * C * S,), tout)
    fn.fnorm_instancenorm(x, g.view, N, C, S, code(torch.bfloat16), code(tout), EPS, None, None)
    torch.cuda.synchronize()
    g.check()
    ref, _, _ = orc.instancenorm_affine(to_f64(x).reshape(N, C, S), None, None, EPS)
    assert_close(to_f64(g.view).reshape(N, C, S), ref, tout, f"case {case}: N={N} C={C} S={S}")


@pytest.mark.parametrize("case", range(CASES))
def test_fuzz_epilogue(orc, case):
    rng = np.random.default_rng(9300 + case)
    C = int(rng.choice([1, 2, 3, 5, 8, 16, 17, 32, 64]))
    S = int(np.exp(rng.uniform(0.0, np.log(200_000))))
    if rng.random() < 0.6:
        S = max(4, S - S % 4)
    N = int(max(1, min(6, 2_000_000 // (S * C))))
    lo = float(rng.uniform(-2.0, 0.0))
    hi = lo + float(rng.uniform(0.0, 3.0))
    x, m = inputs.epilogue(dev(), shape=(N, C, S), seed=9400 + case)
    gy = Guarded((N, S), torch.float32)
    ga = Guarded((N, S), torch.int64)
    fn.fnorm_instancenorm_epilogue(x, m, gy.view, ga.view, N, C, S, EPS, lo, hi)
    torch.cuda.synchronize()
    gy.check()
    ga.check()
    ref, rarg, second = orc.epilogue(x.cpu().numpy(), m.cpu().numpy(), EPS, lo, hi)
    assert_close(gy.view.cpu().numpy(), ref, torch.float32, f"case {case}: N={N} C={C} S={S}")
    a = ga.view.cpu().numpy()
    clear = (ref - second) > 1e-5
    assert np.array_equal(a[clear], rarg[clear]), f"case {case}"
    assert np.all((a >= 0) & (a < C))


@pytest.mark.parametrize("case", range(CASES))
def test_fuzz_batchnorm(orc, case):
    rng = np.random.default_rng(9500 + case)
    S = int(np.exp(rng.uniform(0.0, np.log(60_000))))
    if rng.random() < 0.6:
        S = max(4, S - S % 4)
    C = int(rng.integers(1, 40))
    N = int(max(1, min(16, 2_500_000 // (S * C))))
    if N * S < 2:
        S = 2
    eval_mode = rng.random() < 0.4
    affine = rng.random() < 0.7
    misalign = rng.random() < 0.2
    in_place = rng.random() < 0.2
    x0, g, b, _, _ = inputs.batchnorm(dev(), shape=(N, C, S), seed=9600 + case)
    if not affine:
        g = b = None
    x = _offset_view(N * C * S, torch.float32, misalign, None)
    x.copy_(x0.reshape(-1))
    x = x.view(N, C, S)
    xh = x.cpu().numpy()
    rm = torch.linspace(-0.3, 0.3, C, device=dev())
    rv = torch.linspace(0.4, 1.6, C, device=dev())
    y = x if in_place else _offset_view(N * C * S, torch.float32, misalign).view(N, C, S)
    gh = None if g is None else g.cpu().numpy()
    bh = None if b is None else b.cpu().numpy()
    what = f"case {case}: N={N} C={C} S={S} eval={eval_mode} misalign={misalign} in_place={in_place}"
    if eval_mode:
        ref = orc.batchnorm_eval(xh, gh, bh, 2.0, rm.cpu().numpy(), rv.cpu().numpy(), EPS)
        fn.fnorm_batchnorm_eval(x, y, g, b, 2.0, rm, rv, EPS, N, C, S)
        torch.cuda.synchronize()
        assert_close(y.cpu().numpy(), ref, torch.float32, what)
    else:
        ref, rmo, rvo, _, _ = orc.batchnorm_train(xh, gh, bh, 2.0, rm.cpu().numpy(),
                                                  rv.cpu().numpy(), 0.1, EPS)
        ws = torch.empty(fn.fnorm_batchnorm_workspace_size(N, C, S), dtype=torch.uint8,
                         device=dev())
        fn.fnorm_batchnorm_train(x, y, g, b, 2.0, rm, rv, 0.1, EPS, None, None, N, C, S, ws,
                                 ws.numel())
        torch.cuda.synchronize()
        assert_close(y.cpu().numpy(), ref, torch.float32, what)
        assert np.max(np.abs(rm.cpu().numpy() - rmo)) <= 1e-6, what
        assert np.max(np.abs(rv.cpu().numpy() - rvo)) <= 2e-6, what


@pytest.mark.parametrize("case", range(12))
def test_fuzz_instancenorm_workspace(orc, case):
    """fnorm_instancenorm_ws with few long fp32 slices (the workspace route when
    aligned), random lengths around and above a cluster's capacity, sometimes
    misaligned (then the regular plan), with the mean and rstd outputs."""
    rng = np.random.default_rng(9700 + case)
    S = int(rng.integers(1 << 19, 3 << 20))
    if rng.random() < 0.7:
        S -= S % 4
    NC = int(rng.integers(1, 5))
    misalign = rng.random() < 0.25
    xb = inputs.normal((NC * S + 1,), 9700 + case, dev(), mean=-2.0, std=0.5)
    x = xb[1:] if misalign else xb[:NC * S]
    y = Guarded((NC * S,), torch.float32, offset_elems=1 if misalign else 0)
    mean = torch.empty(NC, device=dev())
    rstd = torch.empty(NC, device=dev())
    nb = fn.fnorm_instancenorm_workspace_size(1, NC, S)
    ws = torch.full((max(nb, 1),), 0x3C, dtype=torch.uint8, device=dev())
    fn.fnorm_instancenorm_ws(x, y.view, 1, NC, S, fn.FNORM_F32, fn.FNORM_F32, EPS, mean, rstd, ws,
                             nb)
    torch.cuda.synchronize()
    y.check()
    ref, rmean, rvar = orc.instancenorm(x.cpu().numpy().reshape(NC, S), EPS)
    assert_close(y.view.cpu().numpy().reshape(NC, S), ref, torch.float32,
                 f"ws case {case} NC={NC} S={S} misalign={misalign}")
    assert np.max(np.abs(mean.cpu().numpy() - rmean)) <= 1e-5
    assert np.allclose(rstd.cpu().numpy(), 1 / np.sqrt(rvar + EPS), rtol=2e-6, atol=0)
