"""The fused epilogue max_c m_c*clamp(IN(x*m_c)) on the GPU through the C ABI
against the oracle: the resident cluster kernel at every cluster size, the
streaming fallback, argmax (bit-exact where the oracle's top two differ),
clamp bounds, odd shapes, guard bands, determinism and the bounded-wait
timeout hook."""
import numpy as np
import pytest
import torch

import normalization_reduction_gb300 as fn
from normalization_reduction_gb300 import inputs
from tests.gpu_util import Guarded, assert_close, dev

pytestmark = pytest.mark.gpu

EPS = 1e-5
ARG_GAP = 1e-5   # argmax compared where the oracle's top-2 gap exceeds this


def run_epi(x, m, lo=-1.0, hi=1.0, eps=EPS, want_arg=True):
    N, C = x.shape[0], x.shape[1]
    S = int(np.prod(x.shape[2:]))
    gy = Guarded((N, S), torch.float32)
    ga = Guarded((N, S), torch.int64) if want_arg else None
    fn.fnorm_instancenorm_epilogue(x, m, gy.view, ga.view if ga else None, N, C, S, eps, lo, hi)
    torch.cuda.synchronize()
    gy.check()
    if ga:
        ga.check()
    return gy.view, (ga.view if ga else None)


def check(orc, x, m, lo=-1.0, hi=1.0, what=""):
    y, arg = run_epi(x, m, lo, hi)
    N, C = x.shape[0], x.shape[1]
    xs = x.cpu().numpy().reshape(N, C, -1)
    ref, rarg, second = orc.epilogue(xs, m.cpu().numpy(), EPS, lo, hi)
    assert_close(y.cpu().numpy(), ref, torch.float32, what)
    a = arg.cpu().numpy()
    clear = (ref - second) > ARG_GAP
    assert np.array_equal(a[clear], rarg[clear]), what
    # where not clearly separated, the chosen channel must still attain the max
    assert np.all((a >= 0) & (a < C))
    return y, arg


def test_page_shape_subset(orc):
    """The page's per-sample shape [16,14,30,30] for 8 samples."""
    x, m = inputs.epilogue(dev(), shape=(8, 16, 14, 30, 30))
    check(orc, x, m, what="page shape")


@pytest.mark.parametrize("cl", [1, 2, 4, 8, 16])
def test_cluster_sizes(orc, fnorm_env, cl):
    """The range kernel at every cluster size."""
    fnorm_env.setenv("FNORM_EPI_CLUSTER", str(cl))
    x, m = inputs.epilogue(dev(), shape=(5, 16, 14, 30, 30))
    check(orc, x, m, what=f"cluster {cl}")


@pytest.mark.parametrize("keep", ["0", "1", "37", "160"])
@pytest.mark.parametrize("shape", [(4, 16, 14, 30, 30), (3, 5, 1000), (2, 1, 4096), (3, 40, 1000),
                                   (2, 9, 4), (2, 3, 2052)])
@pytest.mark.parametrize("cl", ["2", "4"])
def test_l2_keep_sizes(orc, fnorm_env, shape, keep, cl):
    """The L2-form kernel with 0 .. 160 position vectors per channel kept in
    shared memory between its passes (ranges shorter and longer than the kept
    part, kept parts that end inside a tile)."""
    fnorm_env.setenv("FNORM_EPI_KEEP", keep)
    fnorm_env.setenv("FNORM_EPI_CLUSTER", cl)
    x, m = inputs.epilogue(dev(), shape=shape, seed=777 + shape[1])
    check(orc, x, m, what=f"keep {keep} {shape} cl {cl}")


@pytest.mark.parametrize("shape", [(300, 16, 1000), (200, 8, 12600), (513, 3, 256)])
def test_more_samples_than_clusters(orc, shape):
    """More samples than co-resident clusters: each persistent cluster takes
    several samples in turn (alternating exchange slots and barrier phases)."""
    x, m = inputs.epilogue(dev(), shape=shape, seed=600 + shape[0])
    check(orc, x, m, what=f"many samples {shape}")


@pytest.mark.parametrize("shape", [(3, 1, 64), (2, 3, 100), (4, 5, 12), (2, 7, 1000),
                                   (3, 16, 4), (2, 33, 256), (1, 64, 2048), (6, 16, 12600)])
def test_shapes_resident(orc, shape):
    x, m = inputs.epilogue(dev(), shape=shape, seed=1234 + shape[1])
    check(orc, x, m, what=str(shape))


@pytest.mark.parametrize("shape", [(3, 1, 63), (2, 3, 7), (4, 5, 13), (2, 7, 1001),
                                   (2, 16, 12601), (1, 300, 50), (2, 4, 300000)])
def test_shapes_stream(orc, shape):
    """Slices that are not a multiple of 4, or too large for shared memory."""
    x, m = inputs.epilogue(dev(), shape=shape, seed=99 + shape[2])
    check(orc, x, m, what=str(shape))


def test_forced_stream(orc, fnorm_env):
    fnorm_env.setenv("FNORM_EPI_STREAM", "1")
    x, m = inputs.epilogue(dev(), shape=(4, 16, 14, 30, 30))
    check(orc, x, m, what="forced stream")


def test_misaligned_stream(orc):
    N, C, S = 3, 6, 500
    xb, m = inputs.epilogue(dev(), shape=(N, C, S + 1), seed=5)
    flat = xb.reshape(-1)[1:1 + N * C * S]
    x = flat.view(N, C, S)
    check(orc, x, m, what="misaligned")


@pytest.mark.parametrize("lo,hi", [(-1.0, 1.0), (-0.5, 0.25), (0.0, 0.0), (-3.0, 3.0)])
def test_clamp_bounds(orc, lo, hi):
    x, m = inputs.epilogue(dev(), shape=(3, 16, 1000))
    check(orc, x, m, lo, hi, what=f"clamp {lo},{hi}")


def test_ties_lowest_index():
    """Identical channels with identical multipliers tie everywhere."""
    base = torch.randn(2, 1, 4000, device=dev())
    x = base.repeat(1, 5, 1).contiguous()
    m = torch.full((5,), 0.7, device=dev())
    y, arg = run_epi(x, m)
    assert bool((arg == 0).all())


def test_saturated_channels(orc):
    """Outliers clamp to exactly +-1. Since IN(m x) = sign(m) IN(x), a clamped
    outlier contributes m_c * sign(m_c) = |m_c| exactly, so the largest |m_c|
    (channel 2, m = -2) wins there with the value 2.0."""
    N, C, S = 2, 4, 4096
    x = torch.zeros(N, C, S, device=dev())
    x[:, :, 17] = 1000.0
    x[:, :, 18:] = torch.randn(N, C, S - 18, device=dev()) * 0.01
    m = torch.tensor([0.5, 1.5, -2.0, 1.25], device=dev())
    y, arg = check(orc, x, m, what="saturation")
    assert bool((y[:, 17] == 2.0).all()) and bool((arg[:, 17] == 2).all())


def test_deterministic():
    x, m = inputs.epilogue(dev(), shape=(6, 16, 14, 30, 30))
    y1, a1 = run_epi(x, m)
    y2, a2 = run_epi(x, m)
    assert torch.equal(y1, y2) and torch.equal(a1, a2)


def test_no_argmax_output(orc):
    x, m = inputs.epilogue(dev(), shape=(3, 16, 14, 30, 30))
    y, _ = run_epi(x, m, want_arg=False)
    ref, _, _ = orc.epilogue(x.cpu().numpy().reshape(3, 16, -1), m.cpu().numpy(), EPS)
    assert_close(y.cpu().numpy(), ref, torch.float32, "no argmax")


def test_bounded_wait_timeout(orc, fnorm_env):
    """The test hook makes one CTA wait on an mbarrier nothing completes: the
    wait expires after its limit, the error word reports FNORM_ERR_TIMEOUT,
    the context stays usable and the results are still correct."""
    assert fn.fnorm_get_last_error() == fn.Status.OK
    fnorm_env.force_timeout(True)
    x, m = inputs.epilogue(dev(), shape=(2, 16, 14, 30, 30))
    y, arg = run_epi(x, m)
    assert fn.fnorm_get_last_error() == fn.Status.ERR_TIMEOUT
    assert fn.fnorm_get_last_error() == fn.Status.OK   # read-and-clear
    fnorm_env.force_timeout(False)
    ref, _, _ = orc.epilogue(x.cpu().numpy().reshape(2, 16, -1), m.cpu().numpy(), EPS)
    assert_close(y.cpu().numpy(), ref, torch.float32, "after timeout")
    check(orc, x, m, what="after timeout")


def check_no_arg(orc, x, m, lo=-1.0, hi=1.0, what=""):
    """The output without the index (the saturating form of the clamp)
    against the oracle."""
    y, _ = run_epi(x, m, lo, hi, want_arg=False)
    N, C = x.shape[0], x.shape[1]
    ref, _, _ = orc.epilogue(x.cpu().numpy().reshape(N, C, -1), m.cpu().numpy(), EPS, lo, hi)
    assert_close(y.cpu().numpy(), ref, torch.float32, what)
    return y


@pytest.mark.parametrize("lo,hi", [(-1.0, 1.0), (-0.5, 0.25), (0.0, 0.0), (-3.0, 3.0), (0.5, 2.0)])
def test_clamp_bounds_no_index(orc, lo, hi):
    """Both signs of the multiplier (the clamp interval m*[lo, hi] flips for
    m < 0), a zero multiplier and an empty interval, without the index."""
    x, _ = inputs.epilogue(dev(), shape=(3, 16, 1000))
    m = torch.linspace(-1.5, 1.5, 16, device=dev())
    m[7] = 0.0
    check_no_arg(orc, x, m, lo, hi, what=f"clamp {lo},{hi} no index")


def test_saturated_channels_no_index(orc):
    """Clamped outliers without the index: the largest |m_c| wins with 2.0
    (up to the rounding of the saturating clamp)."""
    N, C, S = 2, 4, 4096
    x = torch.zeros(N, C, S, device=dev())
    x[:, :, 17] = 1000.0
    x[:, :, 18:] = torch.randn(N, C, S - 18, device=dev()) * 0.01
    m = torch.tensor([0.5, 1.5, -2.0, 1.25], device=dev())
    y = check_no_arg(orc, x, m, what="saturation, no index")
    assert torch.allclose(y[:, 17], torch.full_like(y[:, 17], 2.0), rtol=0, atol=1e-6)


@pytest.mark.parametrize("S", [4096, 20480, 40000])
@pytest.mark.parametrize("want_arg", [True, False], ids=["index", "no_index"])
@pytest.mark.parametrize("form", ["default", "twopass"])
def test_outliers_at_lane_shifts(orc, fnorm_env, S, want_arg, form):
    """For CTA ranges of at most 1280 vectors (S = 20480 with the default
    4-CTA split: 40 vectors per lane) the statistics are per-lane sums shifted
    by the lane's first value; longer ranges, and every range with
    FNORM_EPI_TWOPASS=1, take exact two-pass tiles. An outlier at the shift is
    the worst case for the shifted sums: put one at the first value of every
    lane of every CTA range, on data with a large offset; the outputs must
    still match the oracle."""
    if form == "twopass":
        fnorm_env.setenv("FNORM_EPI_TWOPASS", "1")
    N, C = 2, 3
    g = torch.Generator().manual_seed(4242 + S)
    x = (torch.randn(N, C, S, generator=g) * 0.5 + 50.0)
    nv4 = S // 4
    per = (nv4 + 3) // 4
    for r in range(4):
        for lane in range(32):
            v = r * per + lane
            if v < min(nv4, (r + 1) * per):
                x[:, :, 4 * v] = 50.0 + 400.0 * (1 if lane % 2 else -1)
    x = x.to(dev())
    m = torch.tensor([0.75, -1.25, 2.0], device=dev())
    if want_arg:
        check(orc, x, m, what=f"lane-shift outliers S={S} {form}")
    else:
        check_no_arg(orc, x, m, what=f"lane-shift outliers S={S} {form} no index")


def _epi_plan(capfd):
    err = capfd.readouterr().err
    lines = [ln for ln in err.splitlines() if "fnorm_instancenorm_epilogue plan" in ln]
    assert lines, err[-2000:]
    return dict(kv.split("=") for kv in lines[-1].split(": ", 1)[1].split())


@pytest.mark.parametrize("C,keep", [(16, 118), (32, 54), (1, 118)])
def test_kept_part_fits_the_carveout_budget(orc, fnorm_env, capfd, C, keep):
    """The L2-form plan keeps as many leading vectors per channel in shared
    memory as fit 33 KB per CTA with its other shared memory (four CTAs per SM
    in the 132 KB shared-memory carveout, the rest of the SM left to L1), at
    most 118: 118 for the page's 16 channels, 54 for 32. The outputs still
    match the oracle."""
    fnorm_env.setenv("FNORM_DEBUG_PLAN", "1")
    x, m = inputs.epilogue(dev(), shape=(3, C, 14, 30, 30))
    check(orc, x, m, what=f"C={C}")
    plan = _epi_plan(capfd)
    assert plan["path"] == "2" and int(plan["cluster"]) == 4
    assert int(plan["keep"]) == keep
    assert int(plan["smem"]) <= 33 * 1024 - 1024 - 64
