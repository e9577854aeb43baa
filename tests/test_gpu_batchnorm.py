"""Training-mode BatchNorm x scale on the GPU through the C ABI against the
oracle: outputs, running-statistic updates, saved statistics, optional
affine terms, element-wise path, in-place use, chunked runs, guard bands,
workspace reuse without clearing, determinism."""
import numpy as np
import pytest
import torch

import normalization_reduction_gb300 as fn
from normalization_reduction_gb300 import inputs
from tests.gpu_util import Guarded, assert_close, dev

pytestmark = pytest.mark.gpu

EPS = 1e-5
MOM = 0.1


def run_bn(x, gamma, beta, rm, rv, scale=2.0, out=None, workspace=None, momentum=MOM):
    N, C = x.shape[0], x.shape[1]
    S = int(np.prod(x.shape[2:])) if x.dim() > 2 else 1
    y = out if out is not None else torch.empty_like(x)
    nbytes = fn.fnorm_batchnorm_workspace_size(N, C, S)
    ws = workspace if workspace is not None else torch.empty(nbytes, dtype=torch.uint8,
                                                             device=x.device)
    sm = torch.empty(C, device=x.device)
    sr = torch.empty(C, device=x.device)
    fn.fnorm_batchnorm_train(x, y, gamma, beta, scale, rm, rv, momentum, EPS, sm, sr, N, C, S, ws,
                             ws.numel())
    torch.cuda.synchronize()
    return y, sm, sr


def check(orc, x, gamma, beta, scale=2.0, with_running=True, what=""):
    C = x.shape[1]
    rm0 = torch.linspace(-0.2, 0.3, C, device=dev())
    rv0 = torch.linspace(0.5, 1.5, C, device=dev())
    rm, rv = (rm0.clone(), rv0.clone()) if with_running else (None, None)
    g = Guarded(tuple(x.shape), torch.float32)
    y, sm, sr = run_bn(x, gamma, beta, rm, rv, scale, out=g.view)
    g.check()
    xs = x.cpu().numpy()
    ref, rmo, rvo, mean, var = orc.batchnorm_train(
        xs.reshape(x.shape[0], C, -1), None if gamma is None else gamma.cpu().numpy(),
        None if beta is None else beta.cpu().numpy(), scale,
        rm0.cpu().numpy() if with_running else None, rv0.cpu().numpy() if with_running else None,
        MOM, EPS)
    assert_close(y.cpu().numpy().reshape(ref.shape), ref, torch.float32, what)
    assert np.max(np.abs(sm.cpu().numpy() - mean)) <= 1e-5, what
    assert np.allclose(sr.cpu().numpy(), 1 / np.sqrt(var + EPS), rtol=2e-6, atol=0), what
    if with_running:
        assert np.max(np.abs(rm.cpu().numpy() - rmo)) <= 1e-6, what
        assert np.max(np.abs(rv.cpu().numpy() - rvo)) <= 2e-6, what
    return y


def test_page_shape_subset(orc):
    """The page's Conv2d output shape [N,64,126,126] at N = 8."""
    x, g, b, _, _ = inputs.batchnorm(dev(), shape=(8, 64, 126, 126))
    check(orc, x, g, b, what="page shape")


@pytest.mark.parametrize("shape", [(2, 3, 1), (1, 2, 2), (3, 4, 5), (2, 3, 4, 4), (5, 7, 33),
                                   (4, 2, 16384), (3, 2, 16385), (2, 3, 40000),
                                   (64, 3, 100), (2, 1, 100003)])
def test_shapes(orc, shape):
    x, g, b, _, _ = inputs.batchnorm(dev(), shape=shape, seed=7 + shape[-1])
    check(orc, x, g, b, what=str(shape))


@pytest.mark.parametrize("shape", [(2, 1, 100000), (300, 3, 4), (5, 7, 36), (1, 200, 16384),
                                   (3, 2, 49152), (9, 64, 15876), (4, 3, 8192), (4, 3, 8196),
                                   (2, 5, 16380)])
@pytest.mark.parametrize("split", ["1", "0"], ids=["split", "registers"])
def test_statistics_kernels(orc, fnorm_env, shape, split):
    """Both vector-mode statistics kernels (registers + TMA staging, registers
    only): runs of many chunks, tiny runs of one vector, units that end in the
    register part, in the staged part and exactly at the chunk size."""
    fnorm_env.setenv("FNORM_BN_SPLIT", split)
    x, g, b, _, _ = inputs.batchnorm(dev(), shape=shape, seed=11 + shape[-1])
    check(orc, x, g, b, what=f"{shape} split={split}")


def test_no_affine_no_running(orc):
    x, _, _, _, _ = inputs.batchnorm(dev(), shape=(4, 6, 300))
    check(orc, x, None, None, scale=1.0, with_running=False, what="plain")


def test_scalar_path(orc, fnorm_env):
    fnorm_env.setenv("FNORM_FORCE_SCALAR", "1")
    x, g, b, _, _ = inputs.batchnorm(dev(), shape=(4, 6, 1000))
    check(orc, x, g, b, what="scalar")


def test_misaligned(orc):
    xb, g, b, _, _ = inputs.batchnorm(dev(), shape=(3, 5, 301))
    x = xb.reshape(-1)[1:1 + 3 * 5 * 300].view(3, 5, 300)
    check(orc, x, g, b, what="misaligned")


def test_in_place(orc):
    x, g, b, _, _ = inputs.batchnorm(dev(), shape=(4, 8, 1000))
    ref, _, _, _, _ = orc.batchnorm_train(x.cpu().numpy(), g.cpu().numpy(), b.cpu().numpy(), 2.0,
                                          None, None, MOM, EPS)
    run_bn(x, g, b, None, None, 2.0, out=x)
    assert_close(x.cpu().numpy(), ref, torch.float32, "in place")


def test_workspace_reuse_dirty(orc):
    """The workspace needs no clearing: fill it with garbage between calls."""
    x, g, b, _, _ = inputs.batchnorm(dev(), shape=(6, 4, 5000))
    nbytes = fn.fnorm_batchnorm_workspace_size(6, 4, 5000)
    ws = torch.full((nbytes,), 0xAB, dtype=torch.uint8, device=dev())
    ref, _, _, _, _ = orc.batchnorm_train(x.cpu().numpy(), g.cpu().numpy(), b.cpu().numpy(), 2.0,
                                          None, None, MOM, EPS)
    for _ in range(2):
        y, _, _ = run_bn(x, g, b, None, None, workspace=ws)
        assert_close(y.cpu().numpy(), ref, torch.float32, "dirty workspace")
        ws.fill_(0x7F)


def test_running_stats_accumulate(orc):
    """Three steps of running-statistic updates match three oracle steps."""
    x, g, b, rm, rv = inputs.batchnorm(dev(), shape=(4, 5, 777))
    rm_h, rv_h = rm.cpu().numpy().astype(np.float64), rv.cpu().numpy().astype(np.float64)
    for step in range(3):
        xs = (x * (1 + step) + step).contiguous()
        run_bn(xs, g, b, rm, rv)
        _, rm_h, rv_h, _, _ = orc.batchnorm_train(xs.cpu().numpy(), g.cpu().numpy(),
                                                  b.cpu().numpy(), 2.0, rm_h, rv_h, MOM, EPS)
    assert np.max(np.abs(rm.cpu().numpy() - rm_h)) <= 1e-5
    assert np.max(np.abs(rv.cpu().numpy() - rv_h)) <= 1e-5


def test_constant_channel_exact():
    x = torch.full((4, 3, 1000), 0.1, device=dev())
    y, sm, _ = run_bn(x, None, None, None, None, scale=1.0)
    assert bool((y == 0).all()) and bool((sm == np.float32(0.1)).all())


def test_deterministic():
    x, g, b, _, _ = inputs.batchnorm(dev(), shape=(16, 8, 3000))
    y1, m1, r1 = run_bn(x, g, b, None, None)
    y2, m2, r2 = run_bn(x, g, b, None, None)
    assert torch.equal(y1, y2) and torch.equal(m1, m2) and torch.equal(r1, r2)


@pytest.mark.parametrize("mode", ["train", "eval"])
def test_bounded_wait_timeout(orc, fnorm_env, mode):
    """The test hook makes one CTA of each staged BatchNorm kernel wait on an
    mbarrier nothing completes: the waits expire, the error word reports
    FNORM_ERR_TIMEOUT (read and cleared) and the results are still correct."""
    assert fn.fnorm_get_last_error() == fn.Status.OK
    x, g, b, _, _ = inputs.batchnorm(dev(), shape=(6, 5, 3000))
    fnorm_env.force_timeout(True)
    if mode == "train":
        y, _, _ = run_bn(x, g, b, None, None)
        ref, _, _, _, _ = orc.batchnorm_train(x.cpu().numpy(), g.cpu().numpy(), b.cpu().numpy(),
                                              2.0, None, None, MOM, EPS)
    else:
        rm = torch.linspace(-0.1, 0.1, 5, device=dev())
        rv = torch.linspace(0.5, 1.5, 5, device=dev())
        y = torch.empty_like(x)
        fn.fnorm_batchnorm_eval(x, y, g, b, 2.0, rm, rv, EPS, 6, 5, 3000)
        torch.cuda.synchronize()
        ref = orc.batchnorm_eval(x.cpu().numpy(), g.cpu().numpy(), b.cpu().numpy(), 2.0,
                                 rm.cpu().numpy(), rv.cpu().numpy(), EPS)
    assert fn.fnorm_get_last_error() == fn.Status.ERR_TIMEOUT
    assert fn.fnorm_get_last_error() == fn.Status.OK
    fnorm_env.force_timeout(False)
    assert_close(y.cpu().numpy(), ref, torch.float32, f"{mode} after timeout")


@pytest.mark.parametrize("shape", [(8, 64, 126, 126), (2, 1, 100000), (300, 3, 4), (5, 7, 36),
                                   (4, 3, 8196), (1, 2, 5), (3, 40, 16384), (64, 3, 100)])
def test_resident_kernel(orc, fnorm_env, shape):
    """The single cooperative launch (statistics, grid barrier, apply with
    each CTA's last unit kept in shared memory) against the oracle: more
    units than CTAs, fewer units than CTAs, units of several chunks, tiny
    units, element-wise fall-back shapes (S % 4 != 0 take the two launches)."""
    fnorm_env.setenv("FNORM_BN_RESIDENT", "1")
    x, g, b, _, _ = inputs.batchnorm(dev(), shape=shape, seed=31 + shape[1])
    check(orc, x, g, b, what=f"resident {shape}")


def test_resident_dirty_workspace_and_repeat(orc, fnorm_env):
    """The barrier counter lives in the caller's workspace, which needs no
    clearing: garbage between calls, and back-to-back calls on one stream."""
    fnorm_env.setenv("FNORM_BN_RESIDENT", "1")
    x, g, b, _, _ = inputs.batchnorm(dev(), shape=(16, 8, 3000))
    nbytes = fn.fnorm_batchnorm_workspace_size(16, 8, 3000)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=dev())
    ref, _, _, _, _ = orc.batchnorm_train(x.cpu().numpy(), g.cpu().numpy(), b.cpu().numpy(), 2.0,
                                          None, None, MOM, EPS)
    for _ in range(3):
        y, _, _ = run_bn(x, g, b, None, None, workspace=ws)
        assert_close(y.cpu().numpy(), ref, torch.float32, "resident, dirty workspace")
        ws.fill_(0x5A)
    y1, _, _ = run_bn(x, g, b, None, None, workspace=ws)
    fnorm_env.delenv("FNORM_BN_RESIDENT")
    y2, _, _ = run_bn(x, g, b, None, None, workspace=ws)
    assert torch.equal(y1, y2)   # same partials, same merge order: same bits as two launches


def test_resident_timeout_hook(orc, fnorm_env):
    fnorm_env.setenv("FNORM_BN_RESIDENT", "1")
    assert fn.fnorm_get_last_error() == fn.Status.OK
    x, g, b, _, _ = inputs.batchnorm(dev(), shape=(6, 5, 3000))
    fnorm_env.force_timeout(True)
    y, _, _ = run_bn(x, g, b, None, None)
    assert fn.fnorm_get_last_error() == fn.Status.ERR_TIMEOUT
    assert fn.fnorm_get_last_error() == fn.Status.OK
    fnorm_env.force_timeout(False)
    ref, _, _, _, _ = orc.batchnorm_train(x.cpu().numpy(), g.cpu().numpy(), b.cpu().numpy(), 2.0,
                                          None, None, MOM, EPS)
    assert_close(y.cpu().numpy(), ref, torch.float32, "resident after timeout")


@pytest.mark.parametrize("shape", [(4096, 64, 1), (1000, 3, 7), (33, 17, 3), (31, 5, 16),
                                   (100000, 2, 1), (1, 2, 16), (2, 1, 1), (65, 300, 2)])
@pytest.mark.parametrize("columns", ["1", "0"], ids=["columns", "units"])
def test_short_runs(orc, fnorm_env, shape, columns):
    """Runs of at most 16 values (BatchNorm over [N, C] and small maps): the
    column form (column statistics over row blocks, channel merge, apply) and
    the per-unit form agree with the oracle, running statistics included."""
    if columns == "0":
        fnorm_env.setenv("FNORM_BN_NO_COLUMNS", "1")
    x, g, b, _, _ = inputs.batchnorm(dev(), shape=shape, seed=41 + shape[0])
    check(orc, x, g, b, what=f"short runs {shape} columns={columns}")

