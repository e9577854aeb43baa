"""InstanceNorm on the GPU through the C ABI against the oracle: every kernel
shape (group, resident, split-resident with TMA staging, stream), vector and element-wise
access, all dtype pairs, ragged and degenerate sizes, misaligned pointers,
in-place use, statistics outputs, determinism and guard bands."""
import numpy as np
import pytest
import torch

import normalization_reduction_gb300 as fn
from normalization_reduction_gb300 import inputs
from tests.gpu_util import Guarded, assert_close, code, dev, to_f64

pytestmark = pytest.mark.gpu

EPS = 1e-5


def run_in(x: torch.Tensor, out_dtype=None, eps=EPS, out=None, stats=False, NC=None, S=None):
    out_dtype = out_dtype or x.dtype
    if S is None:
        S = x.shape[-1]
    if NC is None:
        NC = x.numel() // S if S else 0
    y = out if out is not None else torch.empty(x.shape, dtype=out_dtype, device=x.device)
    mean = torch.empty(max(NC, 1), dtype=torch.float32, device=x.device) if stats else None
    rstd = torch.empty(max(NC, 1), dtype=torch.float32, device=x.device) if stats else None
    fn.fnorm_instancenorm(x, y, 1, NC, S, code(x.dtype), code(out_dtype), eps, mean, rstd)
    torch.cuda.synchronize()
    return y, mean, rstd


def oracle_in(orc, x: torch.Tensor, eps=EPS):
    S = x.shape[-1]
    ref, mean, var = orc.instancenorm(to_f64(x).reshape(-1, S), eps)
    return ref.reshape(x.shape), mean, var


def make_x(NC, S, dtype, seed, dist="normal"):
    if dist == "normal":
        x = inputs.normal((NC, S), seed, "cpu", mean=0.0, std=1.0)
    elif dist == "shifted":
        x = inputs.normal((NC, S), seed, "cpu", mean=3.0, std=2.0)
    else:
        x = inputs.uniform((NC, S), seed, "cpu")
    return x.to(dtype).to(dev())


def test_small_workload(orc):
    """x[2,4,16,16] ~ N(0,1) with slice (1,3) = 5.0: parity and exact zeros."""
    x = inputs.instancenorm_small("cpu")
    xd = x.to(dev())
    y = torch.empty_like(xd)
    fn.fnorm_instancenorm(xd, y, 2, 4, 256, fn.FNORM_F32, fn.FNORM_F32, EPS, None, None)
    torch.cuda.synchronize()
    ref, _, _ = orc.instancenorm(x.numpy().reshape(8, 256), EPS)
    got = y.cpu().numpy().reshape(8, 256)
    assert_close(got, ref, torch.float32, "small")
    assert np.all(got[7] == 0.0) and not np.any(np.signbit(got[7]))


SIZES = [1, 2, 3, 4, 7, 8, 31, 33, 64, 255, 256, 257, 1000, 1024, 2047, 2048, 4097, 12291,
         12600, 16387, 32768, 65536, 100003, 262144]


@pytest.mark.parametrize("S", SIZES)
@pytest.mark.parametrize("dt", ["f32", "bf16", "bf16>f32", "f32>bf16"])
def test_sizes_and_dtypes(orc, S, dt):
    tin = torch.bfloat16 if dt.startswith("bf16") else torch.float32
    tout = {"f32": torch.float32, "bf16": torch.bfloat16, "bf16>f32": torch.float32,
            "f32>bf16": torch.bfloat16}[dt]
    NC = max(3, min(40, 2_000_000 // max(S, 1)))
    x = make_x(NC, S, tin, 10_000 + S, "shifted" if tin == torch.bfloat16 else "normal")
    g = Guarded((NC, S), tout)
    y, mean, rstd = run_in(x, tout, out=g.view, stats=True)
    g.check()
    ref, rmean, rvar = oracle_in(orc, x)
    assert_close(to_f64(y), ref, tout, f"S={S} {dt}")
    assert_close(mean.cpu().numpy()[:NC], rmean, torch.float32, "mean")
    assert np.allclose(rstd.cpu().numpy()[:NC], 1.0 / np.sqrt(rvar + EPS), rtol=2e-6, atol=0)


FORCED = [
    ("group:8:1", [1, 5, 32]), ("group:8:4", [32, 100, 128]), ("group:32:2", [64, 250]),
    ("group:32:4", [7, 512]), ("group:32:8", [1024, 999]),
    ("resident:128:4", [1, 2048, 1500]), ("resident:256:4", [4096, 333]),
    ("resident:256:8", [8192, 6000]), ("resident:512:8", [16384, 9999]),
    ("resident:1024:8", [32768, 20000]),
    ("resident:128:4:3", [5000, 6144, 1]), ("resident:256:8:2", [8193, 16384]),
    ("resident:512:8:8", [131072, 70000]), ("resident:1024:8:4", [131072, 100001]),
    ("resident:512:8:16", [262144, 200000]), ("resident:1024:8:16", [524288]),
    ("split:128:8:8:1", [8192, 4000, 16]), ("split:256:8:8:1", [16384, 10000, 64]),
    ("split:512:8:8:1", [32768, 65536, 20000]), ("split:1024:8:8:1", [65536, 131072, 40000]),
    ("split:512:8:8:3", [40000, 96000, 8]), ("split:512:8:8:8", [262144, 200000]),
    ("split:512:8:8:16", [524288, 1048576]), ("split:1024:8:8:8", [524288, 1000000]),
    ("split:256:8:0:1", [8192, 104]), ("split:512:8:0:4", [65536, 50000]),
    ("split:1024:8:0:8", [262144]),
    ("stream:1", [1, 77777]), ("stream:2", [12600, 3]), ("stream:8", [262144, 99999]),
    ("stream:16", [600000]),
]


@pytest.mark.parametrize("path,sizes", FORCED, ids=[p for p, _ in FORCED])
@pytest.mark.parametrize("scalar", [False, True], ids=["vec", "scalar"])
def test_forced_paths(orc, fnorm_env, path, sizes, scalar):
    """Every kernel shape, including empty CTAs in a cluster and 16-CTA clusters."""
    parts = path.split(":")
    if parts[0] == "split" and scalar:
        pytest.skip("the split kernel has vector access only")
    if parts[0] in ("resident", "split") and len(parts) >= 4:
        forced = path
    elif parts[0] == "resident":
        forced = path + ":1"
    else:
        forced = path
    fnorm_env.setenv("FNORM_FORCE_PATH", forced)
    if scalar:
        fnorm_env.setenv("FNORM_FORCE_SCALAR", "1")
    for S in sizes:
        for tin in (torch.float32, torch.bfloat16):
            W = 4 if tin == torch.float32 else 8
            slots = -(-S // W)
            if parts[0] == "group" and int(parts[1]) * int(parts[2]) < slots:
                continue
            if parts[0] == "resident":
                cl = int(forced.split(":")[3])
                if int(parts[1]) * int(parts[2]) * cl < slots:
                    continue
            if parts[0] == "split":
                if int(parts[1]) * (int(parts[2]) + int(parts[3])) * int(parts[4]) < slots:
                    continue
                if S % W:
                    continue
            NC = max(2, min(24, 3_000_000 // S))
            x = make_x(NC, S, tin, 20_000 + S, "shifted")
            y, _, _ = run_in(x, tin)
            ref, _, _ = oracle_in(orc, x)
            assert_close(to_f64(y), ref, tin, f"{forced} S={S} {tin}")


@pytest.mark.parametrize("S", [256, 12600, 262144])
def test_misaligned_pointers(orc, S):
    """Base pointers one element off a 16-byte boundary take the element-wise path."""
    for tin, off in ((torch.float32, 1), (torch.bfloat16, 1), (torch.bfloat16, 3)):
        NC = 5
        buf = make_x(NC * S + off, 1, tin, 33_000 + S).reshape(-1)
        x = buf[off:off + NC * S].view(NC, S)
        g = Guarded((NC, S), tin, offset_elems=off)
        y, _, _ = run_in(x, tin, out=g.view)
        g.check()
        ref, _, _ = oracle_in(orc, x)
        assert_close(to_f64(y), ref, tin, f"misaligned S={S}")


def test_in_place(orc):
    x = make_x(20, 4096, torch.float32, 44)
    ref, _, _ = oracle_in(orc, x)
    fn.fnorm_instancenorm(x, x, 4, 5, 4096, fn.FNORM_F32, fn.FNORM_F32, EPS, None, None)
    torch.cuda.synchronize()
    assert_close(to_f64(x), ref, torch.float32, "in place")


@pytest.mark.parametrize("S,dt,NC", [(262144, torch.float32, 80), (65536, torch.bfloat16, 400),
                                     (200, torch.bfloat16, 3000), (600000, torch.float32, 5),
                                     (12600, torch.float32, 700)])
def test_in_place_every_family(orc, S, dt, NC):
    """y == x for the split kernel (registers + staged part prefetched for the
    next slice, 16-CTA clusters, more slices than clusters), the group kernel
    and the stream form: every slice is read before it is written."""
    x = make_x(NC, S, dt, 45 + S)
    ref, _, _ = oracle_in(orc, x)
    c = code(dt)
    fn.fnorm_instancenorm(x, x, 1, NC, S, c, c, EPS, None, None)
    torch.cuda.synchronize()
    assert_close(to_f64(x), ref, dt, f"in place S={S}")


def test_constant_slices_exact_zero():
    """Constant slices of awkward values (not exactly summable) give exact zeros."""
    for S in (3, 1000, 12600, 262144):
        for v in (5.0, 0.1, -3.7e5, 1e-30):
            x = torch.full((3, S), v, dtype=torch.float32, device=dev())
            y, mean, _ = run_in(x, stats=True)
            assert bool((y == 0).all()), (S, v)
            assert bool((mean[:3] == np.float32(v)).all()), (S, v)


def test_uniform_input(orc):
    """The page's own test input, torch.rand ~ U[0,1), at a reduced batch."""
    x = make_x(64, 512 * 512, torch.float32, 55, "uniform")
    y, _, _ = run_in(x)
    ref, _, _ = oracle_in(orc, x)
    assert_close(to_f64(y), ref, torch.float32, "uniform")


def test_deterministic():
    for S in (256, 12600, 262144, 600000):
        x = make_x(12, S, torch.float32, 66 + S)
        y1, m1, _ = run_in(x, stats=True)
        y2, m2, _ = run_in(x, stats=True)
        assert torch.equal(y1, y2) and torch.equal(m1, m2), S


def test_empty_and_eps_zero():
    x = torch.empty((0, 16), device=dev())
    y, _, _ = run_in(x, NC=0, S=16)
    z = torch.randn(4, 100, device=dev())
    y, _, _ = run_in(z, eps=0.0)
    assert bool(torch.isfinite(y).all())


def test_mixed_scale_slices(orc):
    """Slices with very different scales and offsets in one call."""
    S = 4096
    base = make_x(8, S, torch.float32, 77)
    scales = torch.tensor([1e-3, 1.0, 1e3, 1e-2, 50.0, 7.0, 1e4, 0.5], device=dev()).view(8, 1)
    shifts = torch.tensor([0.0, 100.0, -1e3, 5.0, 1e4, -7.0, 3.0, 1e2], device=dev()).view(8, 1)
    x = (base * scales + shifts).contiguous()
    y, _, _ = run_in(x)
    ref, _, _ = oracle_in(orc, x)
    assert_close(to_f64(y), ref, torch.float32, "mixed scales")


def test_bounded_wait_timeout(orc, fnorm_env):
    """The test hook makes one CTA of the split kernel wait, after its last
    cluster barrier, on an mbarrier nothing completes: the wait expires after
    its limit, the error word reports FNORM_ERR_TIMEOUT (read and cleared), the
    context stays usable and the results are correct."""
    assert fn.fnorm_get_last_error() == fn.Status.OK
    fnorm_env.force_timeout(True)
    x = make_x(48, 200000, torch.float32, 515)   # split kernel, 2-CTA clusters
    y, _, _ = run_in(x)
    assert fn.fnorm_get_last_error() == fn.Status.ERR_TIMEOUT
    assert fn.fnorm_get_last_error() == fn.Status.OK
    fnorm_env.force_timeout(False)
    ref, _, _ = oracle_in(orc, x)
    assert_close(to_f64(y), ref, torch.float32, "after timeout")
    y2, _, _ = run_in(x)
    assert torch.equal(y, y2)


@pytest.mark.parametrize("shape,dt", [((1, 3, 2048, 2048), torch.float32),
                                      ((2, 1, 1500, 1500), torch.bfloat16),
                                      ((1, 1, 1 << 21, 1), torch.bfloat16)])
def test_few_long_slices(orc, shape, dt):
    """A few slices longer than a cluster holds (the stream form; 16-CTA
    clusters when 8 would leave most SMs idle), in the default plan."""
    N, C = shape[0], shape[1]
    S = shape[2] * shape[3]
    x = make_x(N * C, S, dt, 77 + S)
    y, _, _ = run_in(x, dt)
    ref, _, _ = oracle_in(orc, x)
    assert_close(to_f64(y), ref, dt, f"few long slices {shape}")


PACKED_CASES = [(3, 1 << 20, None), (2, 1047776, None), (3, 300000, "split:256:8:8:12"),
                (2, 600000, "split:512:8:8:10"), (4, 262144, None),
                (300, 4096, None), (37, 3000, None), (5, 2056, None)]


@pytest.mark.parametrize("NC,S,path", PACKED_CASES,
                         ids=[f"{n}x{s}-{p or 'default'}" for n, s, p in PACKED_CASES])
@pytest.mark.parametrize("tout", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("dist", ["normal", "shifted"])
def test_bf16_packed_matches_scalar(orc, fnorm_env, NC, S, path, tout, dist):
    """bf16 slices spread over clusters of more than 8 CTAs, and slices of
    2049-4096 values held by one 64-thread CTA, take one pass of shifted sums
    and packed pair arithmetic (two fp32 lanes per instruction);
    FNORM_NO_PACK=1 gives the exact two-pass scalar loops. Both must match the
    oracle (outputs, means, rstd) and each other within the tolerance. The
    case S = 262144 (8-CTA clusters) runs the scalar loops both times and must
    be bit-identical. S = 4096 fills every thread's slots (equal-count merges);
    3000 and 2056 leave threads partly or wholly empty."""
    if path:
        fnorm_env.setenv("FNORM_FORCE_PATH", path)
    x = make_x(NC, S, torch.bfloat16, 5150 + S % 997, dist)
    y1, m1, r1 = run_in(x, out_dtype=tout, stats=True)
    fnorm_env.setenv("FNORM_NO_PACK", "1")
    y2, m2, r2 = run_in(x, out_dtype=tout, stats=True)
    ref, rmean, rvar = oracle_in(orc, x)
    for y, m, r, what in ((y1, m1, r1, "packed"), (y2, m2, r2, "scalar")):
        assert_close(to_f64(y), ref, tout, f"{what} {NC}x{S} {path} {dist}")
        assert np.max(np.abs(m.cpu().numpy()[:NC] - rmean)) <= 1e-5 * (1 + np.max(np.abs(rmean)))
        assert np.allclose(r.cpu().numpy()[:NC], 1 / np.sqrt(rvar + EPS), rtol=2e-6, atol=0)
    if S == 262144:
        assert torch.equal(y1, y2) and torch.equal(m1, m2) and torch.equal(r1, r2)


@pytest.mark.parametrize("S,threads,chunk", [(1 << 20, 512, 8192), (1 << 19, 256, 4096),
                                             (4096, 64, 512)])
def test_bf16_packed_outliers_at_thread_shifts(orc, S, threads, chunk):
    """The packed form's one-pass sums are shifted by each thread's first value
    (its first staged vector, or its first register vector when the CTA stages
    nothing: vector r*chunk + t of CTA r's chunk, element 0).
    An outlier there is their worst case: put one at every thread's shift, on
    data with a large offset, and compare with the oracle (fp32 output)."""
    NC = 2
    g = torch.Generator().manual_seed(777 + S)
    x = torch.randn(NC, S, generator=g) * 0.5 + 3.0
    nvec = S // 8
    for r in range((nvec + chunk - 1) // chunk):
        for t in range(threads):
            v = r * chunk + t
            if v < nvec:
                x[:, 8 * v] = 3.0 + (400.0 if t % 2 else -400.0)
    x = x.to(torch.bfloat16).to(dev())
    y, m, rs = run_in(x, out_dtype=torch.float32, stats=True)
    ref, rmean, rvar = oracle_in(orc, x)
    assert_close(to_f64(y), ref, torch.float32, f"thread-shift outliers S={S}")
    assert np.allclose(rs.cpu().numpy()[:NC], 1 / np.sqrt(rvar + EPS), rtol=2e-6, atol=0)


@pytest.mark.parametrize("shape,dtype", [
    ((1, 1, 4096, 4100), torch.float32),   # one slice of 16.8 M values: the workspace route
    ((1, 3, 2048, 2048), torch.float32),
    ((8, 3, 1024, 1024), torch.float32),   # 24 slices
    ((1, 1, 2048, 2050), torch.bfloat16),  # bf16 keeps fnorm_instancenorm's plan
    ((2, 3, 64, 64), torch.float32),       # fits a cluster: fnorm_instancenorm's plan
])
def test_workspace_entry_point(orc, shape, dtype):
    """fnorm_instancenorm_ws against the oracle, element by element, with the
    mean and rstd outputs, on shapes that take its workspace route (few fp32
    slices longer than a cluster holds) and shapes that do not; the workspace
    starts dirty."""
    N, C = shape[0], shape[1]
    S = int(np.prod(shape[2:]))
    x = inputs.normal((N, C, S), 1301 + C, dev(), mean=1.5, std=2.0, dtype=dtype)
    y = torch.empty_like(x)
    mean = torch.empty(N * C, device=dev())
    rstd = torch.empty(N * C, device=dev())
    nb = fn.fnorm_instancenorm_workspace_size(N, C, S)
    ws = torch.full((max(nb, 1),), 0xA5, dtype=torch.uint8, device=dev())
    code = fn.FNORM_F32 if dtype == torch.float32 else fn.FNORM_BF16
    fn.fnorm_instancenorm_ws(x, y, N, C, S, code, code, EPS, mean, rstd, ws, nb)
    torch.cuda.synchronize()
    assert fn.fnorm_get_last_error() == fn.Status.OK
    if dtype == torch.float32:
        ref, rmean, rvar = orc.instancenorm(x.cpu().numpy().reshape(N * C, S), EPS)
        assert_close(y.cpu().numpy().reshape(N * C, S), ref, torch.float32, f"ws {shape}")
    else:
        xb = x.view(torch.int16).cpu().numpy().view(np.uint16).reshape(N * C, S)
        ref_bits, rmean, rvar = orc.instancenorm(xb, EPS)
        yb = y.view(torch.int16).cpu().numpy().view(np.uint16).reshape(N * C, S)
        to64 = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        assert_close(to64(yb), to64(ref_bits), torch.bfloat16, f"ws {shape}")
    assert np.max(np.abs(mean.cpu().numpy() - rmean)) <= 1e-5
    assert np.allclose(rstd.cpu().numpy(), 1 / np.sqrt(rvar + EPS), rtol=2e-6, atol=0)
    if shape == (1, 1, 4096, 4100):
        assert nb > 0
        with pytest.raises(fn.FnormError) as e:   # too small a workspace
            fn.fnorm_instancenorm_ws(x, y, N, C, S, code, code, EPS, None, None, ws, nb - 256)
        assert e.value.status == fn.Status.ERR_INVALID_ARG


@pytest.mark.parametrize("shape", [(1, 1, 4096, 4100), (1, 3, 2048, 2048), (8, 3, 1024, 1024),
                                   (38, 1, 1024, 1024), (2, 1, 1000, 1004)])
def test_long_slices_without_workspace(orc, fnorm_env, capfd, shape):
    """fnorm_instancenorm (no workspace) on few fp32 slices longer than a
    cluster holds, out of place: the output buffer carries the per-unit
    statistics between its launches. Element-wise against the oracle with the
    mean and rstd outputs and guard bands around y; y starts dirty. The plan
    line shows the route; with more than 1024 units per slice the result is
    the workspace route's bit for bit (same kernels, same merge order). An
    in-place call on the same shape takes the cluster stream and still
    matches."""
    N, C = shape[0], shape[1]
    S = int(np.prod(shape[2:]))
    fnorm_env.setenv("FNORM_DEBUG_PLAN", "1")
    x = inputs.normal((N, C, S), 1401 + C, dev(), mean=-2.5, std=3.0)
    g = Guarded((N, C, S), torch.float32)
    g.view.fill_(float("nan"))
    mean = torch.empty(N * C, device=dev())
    rstd = torch.empty(N * C, device=dev())
    fn.fnorm_instancenorm(x, g.view, N, C, S, fn.FNORM_F32, fn.FNORM_F32, EPS, mean, rstd)
    torch.cuda.synchronize()
    g.check()
    assert fn.fnorm_get_last_error() == fn.Status.OK
    assert "route=output_scratch" in capfd.readouterr().err
    ref, rmean, rvar = orc.instancenorm(x.cpu().numpy().reshape(N * C, S), EPS)
    assert_close(g.view.cpu().numpy().reshape(N * C, S), ref, torch.float32, f"no ws {shape}")
    assert np.max(np.abs(mean.cpu().numpy() - rmean)) <= 1e-5
    assert np.allclose(rstd.cpu().numpy(), 1 / np.sqrt(rvar + EPS), rtol=2e-6, atol=0)
    if S // 16384 >= 1024:
        nb = fn.fnorm_instancenorm_workspace_size(N, C, S)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev())
        y2 = torch.empty_like(x)
        fn.fnorm_instancenorm_ws(x, y2, N, C, S, fn.FNORM_F32, fn.FNORM_F32, EPS, None, None,
                                 ws, nb)
        torch.cuda.synchronize()
        assert torch.equal(y2, g.view)
    xi = x.clone()
    fn.fnorm_instancenorm(xi, xi, N, C, S, fn.FNORM_F32, fn.FNORM_F32, EPS, None, None)
    torch.cuda.synchronize()
    assert "route=output_scratch" not in capfd.readouterr().err
    assert_close(xi.cpu().numpy().reshape(N * C, S), ref, torch.float32, f"in place {shape}")


@pytest.mark.parametrize("shape", [(1, 3, 2048, 2048), (8, 3, 1024, 1024), (2, 1, 1000, 1004)])
def test_long_slices_affine_without_workspace(orc, fnorm_env, capfd, shape):
    """The affine form on few long fp32 slices takes the same three-launch
    route (gamma/beta of slice q = n*C + c are those of channel c): against
    the oracle's affine InstanceNorm, with the statistics outputs; in place it
    takes the cluster stream and matches too."""
    N, C = shape[0], shape[1]
    S = int(np.prod(shape[2:]))
    fnorm_env.setenv("FNORM_DEBUG_PLAN", "1")
    x = inputs.normal((N, C, S), 1701 + C, dev(), mean=1.0, std=0.5)
    gamma, beta = inputs.channel_affine(C, 1702, dev())
    y = torch.full_like(x, float("nan"))
    mean = torch.empty(N * C, device=dev())
    rstd = torch.empty(N * C, device=dev())
    fn.fnorm_instancenorm_affine(x, y, gamma, beta, N, C, S, fn.FNORM_F32, fn.FNORM_F32, EPS,
                                 mean, rstd)
    torch.cuda.synchronize()
    assert "route=output_scratch" in capfd.readouterr().err
    ref, rmean, rvar = orc.instancenorm_affine(x.cpu().numpy().astype(np.float64),
                                               gamma.cpu().numpy(), beta.cpu().numpy(), EPS)
    assert_close(y.cpu().numpy(), ref, torch.float32, f"affine no ws {shape}")
    assert np.max(np.abs(mean.cpu().numpy() - np.asarray(rmean).reshape(-1))) <= 1e-5
    assert np.allclose(rstd.cpu().numpy(), 1 / np.sqrt(np.asarray(rvar).reshape(-1) + EPS),
                       rtol=2e-6, atol=0)
    xi = x.clone()
    fn.fnorm_instancenorm_affine(xi, xi, gamma, beta, N, C, S, fn.FNORM_F32, fn.FNORM_F32, EPS,
                                 None, None)
    torch.cuda.synchronize()
    assert "route=output_scratch" not in capfd.readouterr().err
    assert_close(xi.cpu().numpy(), ref, torch.float32, f"affine in place {shape}")


def test_injected_launch_failure_leaves_outputs_untouched(orc):
    """A call failed by fnorm_debug_fail_launches raises FNORM_ERR_CUDA and
    writes nothing; the next call runs normally."""
    x = inputs.normal((3, 4, 1000), 1501, dev())
    g = Guarded((3, 4, 1000), torch.float32)
    fn.fnorm_debug_fail_launches(1)
    try:
        with pytest.raises(fn.FnormError) as e:
            fn.fnorm_instancenorm(x, g.view, 3, 4, 1000, fn.FNORM_F32, fn.FNORM_F32, EPS, None,
                                  None)
        assert e.value.status == fn.Status.ERR_CUDA
        torch.cuda.synchronize()
        assert bool((g.buf == g.buf[0]).all())          # canary value everywhere
        fn.fnorm_instancenorm(x, g.view, 3, 4, 1000, fn.FNORM_F32, fn.FNORM_F32, EPS, None, None)
        torch.cuda.synchronize()
    finally:
        fn.fnorm_debug_fail_launches(0)
    g.check()
    ref, _, _ = orc.instancenorm(x.cpu().numpy().reshape(12, 1000), EPS)
    assert_close(g.view.cpu().numpy().reshape(12, 1000), ref, torch.float32, "after injected")


@pytest.mark.parametrize("in_place", [False, True], ids=["out_of_place", "in_place"])
def test_torch_helper_long_slices(orc, in_place):
    """The torch helper instance_norm on few long fp32 slices: out of place it
    calls fnorm_instancenorm (statistics kept in y), in place
    fnorm_instancenorm_ws with a workspace it allocates; both match the
    oracle, with the statistics outputs."""
    N, C, S = 1, 2, 1 << 20
    x = inputs.normal((N, C, 1024, 1024), 1601, dev(), mean=0.5, std=1.5)
    ref, rmean, rvar = orc.instancenorm(x.cpu().numpy().reshape(N * C, S), EPS)
    xin = x.clone() if in_place else x
    y, mean, rstd = fn.instance_norm(xin, out=xin if in_place else None, return_stats=True)
    torch.cuda.synchronize()
    if in_place:
        assert y.data_ptr() == xin.data_ptr()
    assert_close(y.cpu().numpy().reshape(N * C, S), ref, torch.float32, "helper")
    assert np.max(np.abs(mean.cpu().numpy() - rmean)) <= 1e-5
    assert np.allclose(rstd.cpu().numpy(), 1 / np.sqrt(rvar + EPS), rtol=2e-6, atol=0)
