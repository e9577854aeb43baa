"""Pins for the oracle: checks against what the pages and mathematics fix.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError on
a mismatch. ``test_oracle_pins.py`` runs them on the real oracle;
``test_oracle_mutants.py`` runs them on copies of the oracle with one planted
mistake each and requires every mutant to fail at least one pin.

Kinds of pin used here (none re-types the oracle's own formula):
* exact rational arithmetic (``fractions`` + ``decimal``) on tiny integer inputs;
* closed forms (two-valued slices, affine images, clamp saturation);
* independent library routines (torch's float64 CPU instance_norm / batch_norm,
  numpy's mean/var);
* page-stated facts from ``tests/golden/page_facts.txt``.
"""
from __future__ import annotations

import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import torch
import torch.nn.functional as F

from normalization_reduction_gb300 import inputs

EPS = 1e-5
EPS_Q = Fraction(1, 100000)
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
getcontext().prec = 60


def read_facts(name: str = "page_facts.txt") -> dict:
    """key = value lines; '#' starts a comment (the citation)."""
    facts = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            facts[k] = v
    return facts


def _exact_in(vals, eps_q=EPS_Q):
    """Exact InstanceNorm of one slice: returns (mean, var, [y as Decimal])."""
    q = [Fraction(v) for v in vals]
    n = len(q)
    mean = sum(q) / n
    var = sum((v - mean) ** 2 for v in q) / n
    denom = (Decimal(var.numerator) / Decimal(var.denominator)
             + Decimal(eps_q.numerator) / Decimal(eps_q.denominator)).sqrt()
    ys = [(Decimal((v - mean).numerator) / Decimal((v - mean).denominator)) / denom for v in q]
    return mean, var, ys


def _close(a, b, rel=1e-14, abs_=1e-300):
    return abs(float(a) - float(b)) <= max(abs_, rel * abs(float(b)))


# ---------------------------------------------------------------------------
# InstanceNorm
# ---------------------------------------------------------------------------
HAND_SLICES = [
    [1, 2, 3, 4],          # mean 5/2, var 5/4
    [-3, 0, 0, 3],         # mean 0, var 9/2
    [5, 5, 5, 5],          # constant -> exact zeros
    [0, 0, 0, 8],          # mean 2, var 12
    [7, -1, 2, 2],         # mean 5/2, var 33/4
    [1000, 1001, 999, 1000],
    [-2, -2, 6, 6],
    [3, 1, 4, 1],
]


def pin_instancenorm_exact_rationals(orc):
    """2x2x2x2-sized hand cases (4 values per slice) against exact arithmetic."""
    x = np.array(HAND_SLICES, dtype=np.float64).reshape(2, 4, 2, 2)
    y, mean, var = orc.instancenorm(x.reshape(8, 4), EPS)
    for i, vals in enumerate(HAND_SLICES):
        em, ev, ey = _exact_in(vals)
        assert _close(mean[i], em), (i, mean[i], em)
        assert _close(var[i], ev), (i, var[i], ev)
        for j in range(4):
            assert abs(y[i, j] - float(ey[j])) <= 4e-16 * max(1.0, abs(float(ey[j]))), (i, j)
    # the worked example {1,2,3,4}: mean 2.5, biased var 1.25 (not 5/3 unbiased)
    assert mean[0] == 2.5 and var[0] == 1.25


def pin_instancenorm_f32_rounding(orc):
    """The fp32 output is the exact result rounded once (within one fp32 ulp)."""
    x = np.array(HAND_SLICES, dtype=np.float32)
    y32, _, _ = orc.instancenorm(x, EPS)
    for i, vals in enumerate(HAND_SLICES):
        _, _, ey = _exact_in(vals)
        for j in range(4):
            e = float(ey[j])
            assert abs(float(y32[i, j]) - e) <= np.spacing(np.float32(abs(e)) + np.float32(0)), (i, j)


def pin_instancenorm_two_valued_closed_form(orc):
    """A slice holding b+a and b-a equally often has mean b and variance a^2,
    so every output is exactly +-a/sqrt(a^2+eps)."""
    rng = np.random.default_rng(7)
    for a, b, S in ((2.0, 3.0, 64), (0.5, -7.25, 1024), (2.0 ** -10, 1.0, 256), (96.0, 0.0, 2)):
        sgn = np.where(rng.permutation(S) % 2 == 0, 1.0, -1.0)
        x = (b + a * sgn).reshape(1, S)
        y, mean, var = orc.instancenorm(x, EPS)
        assert mean[0] == b and abs(var[0] - a * a) <= 1e-15 * a * a
        expect = a / math.sqrt(a * a + EPS)
        assert np.all(np.abs(y[0] - sgn * expect) <= 1e-15 * expect), (a, b, S)


def pin_instancenorm_output_moments(orc):
    """Output mean is 0 and output biased variance is var/(var+eps)."""
    rng = np.random.default_rng(11)
    x = rng.integers(-1000, 1000, size=(6, 4096)).astype(np.float64) / 8.0
    y, _, _ = orc.instancenorm(x, EPS)
    for i in range(6):
        v = float(np.var(x[i]))  # numpy pairwise-summation routine, not the oracle
        assert abs(float(np.mean(y[i]))) <= 1e-12
        assert abs(float(np.var(y[i])) - v / (v + EPS)) <= 1e-12


def pin_instancenorm_vs_torch(orc):
    """torch.nn.functional.instance_norm in float64 on the CPU (library routine)."""
    x = torch.randn(3, 5, 7, 9, generator=torch.Generator().manual_seed(5), dtype=torch.float64)
    x = x * torch.linspace(0.1, 4.0, 5, dtype=torch.float64).view(1, 5, 1, 1) + 2.5
    ref = F.instance_norm(x, eps=EPS).numpy()
    y, mean, var = orc.instancenorm(x.numpy().reshape(15, 63), EPS)
    assert np.max(np.abs(y.reshape(ref.shape) - ref)) <= 1e-12
    xs = x.numpy().reshape(15, 63)
    assert np.max(np.abs(mean - xs.mean(axis=1))) <= 1e-13
    assert np.max(np.abs(var - xs.var(axis=1))) <= 1e-12


def pin_instancenorm_constant_slice(orc):
    """The small workload's slice (1,3) is the constant 5.0: all exact zeros;
    the other slices match the library routine."""
    x = inputs.instancenorm_small("cpu")
    shape = tuple(x.shape)
    y, _, _ = orc.instancenorm(x.numpy().reshape(-1, shape[2] * shape[3]), EPS)
    y = y.reshape(shape)
    assert np.all(y[1, 3] == 0.0) and not np.any(np.signbit(y[1, 3]))
    ref = F.instance_norm(x.double(), eps=EPS).float().numpy()
    mask = np.ones(shape[:2], dtype=bool)
    mask[1, 3] = False
    assert np.max(np.abs(y[mask] - ref[mask])) <= 1e-6


def pin_instancenorm_affine_image(orc):
    """IN(a x + b) = a (x - mu) / sqrt(a^2 var + eps): the closed form that the
    epilogue's pre-multiplier relies on; negative a flips the sign."""
    vals = [3, -1, 4, 1, -5, 9, 2, -6]
    mu = Fraction(sum(vals), len(vals))
    var = sum((Fraction(v) - mu) ** 2 for v in vals) / len(vals)
    for a, b in ((3, 7), (-2, 1), (1, -100)):
        x = np.array([[a * v + b for v in vals]], dtype=np.float64)
        y, _, _ = orc.instancenorm(x, EPS)
        d = (Decimal(a * a) * Decimal(var.numerator) / Decimal(var.denominator)
             + Decimal(1) / Decimal(100000)).sqrt()
        for j, v in enumerate(vals):
            num = Fraction(a) * (Fraction(v) - mu)
            e = Decimal(num.numerator) / Decimal(num.denominator) / d
            assert abs(y[0, j] - float(e)) <= 1e-15, (a, b, j)


def pin_instancenorm_degenerate_shapes(orc):
    """S == 1 gives exact zeros (the lone value is the mean); NC == 0 is empty."""
    y, mean, var = orc.instancenorm(np.array([[3.5], [-2.0]]), EPS)
    assert np.all(y == 0.0) and list(mean) == [3.5, -2.0] and list(var) == [0.0, 0.0]
    y, _, _ = orc.instancenorm(np.zeros((0, 8)), EPS)
    assert y.shape == (0, 8)


def pin_instancenorm_bf16(orc):
    """bf16 path: inputs exact, output = nearest-even bf16 of the exact result."""
    rng = np.random.default_rng(3)
    xf = (rng.standard_normal((4, 256)) * 2 + 3).astype(np.float32)
    xb = torch.from_numpy(xf).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    yb, mean, var = orc.instancenorm(bits, EPS)
    x64 = xb.double()
    ref = F.instance_norm(x64.unsqueeze(0), eps=EPS).squeeze(0).numpy()
    assert np.max(np.abs(mean - x64.numpy().mean(axis=1))) <= 1e-13
    ref_bits = orc.round_bf16(ref)
    # identical except where the library value sits within 1e-12 of a rounding tie
    assert np.mean(ref_bits == yb) > 0.999
    assert np.max(np.abs(orc.bf16_to_f64(yb) - ref)) <= 2.0 ** -8 * np.max(np.abs(ref))


# ---------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------
def pin_bf16_rounding(orc):
    """Against torch's float32->bfloat16 cast (exact for fp32-representable
    inputs), plus hand ties-to-even cases."""
    rng = np.random.default_rng(9)
    f = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),   # subnormals
        (rng.standard_normal(2000) * 1e37).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38], dtype=np.float32),
    ])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.round_bf16(f.astype(np.float64))
    assert np.array_equal(got, ref)
    # ties: 1 + 2^-8 -> 1 (even); 1 + 3*2^-8 -> 1 + 2^-6 (even); just above a tie -> up
    cases = {1 + 2.0 ** -8: 0x3F80, 1 + 3 * 2.0 ** -8: 0x3F82, 1 + 2.0 ** -8 + 2.0 ** -40: 0x3F81,
             -(1 + 2.0 ** -8): 0xBF80, 2.0 ** 128: 0x7F80, 3.0e38 * 1.2: 0x7F80}
    got = orc.round_bf16(np.array(list(cases), dtype=np.float64))
    assert [int(v) for v in got] == list(cases.values())


# ---------------------------------------------------------------------------
# Fused epilogue
# ---------------------------------------------------------------------------
def _epilogue_torch(x64: torch.Tensor, m64: torch.Tensor, lo=-1.0, hi=1.0):
    """The page's module chain, each op a torch float64 CPU routine."""
    bs = (1, -1) + (1,) * (x64.dim() - 2)
    v = x64 * m64.view(bs)
    t = F.instance_norm(v, eps=EPS)
    z = torch.clamp(t, lo, hi) * m64.view(bs)
    return z


def pin_epilogue_vs_torch(orc):
    g = torch.Generator().manual_seed(21)
    x = (torch.randn(3, 5, 4, 6, 7, generator=g) * 1.3 + 0.2).float()
    m = torch.randn(5, generator=g).float()
    y, arg, second = orc.epilogue(x.numpy(), m.numpy(), EPS)
    z = _epilogue_torch(x.double(), m.double()).float()   # fp32 decision precision
    zmax, zarg = z.max(dim=1)
    assert np.array_equal(y, zmax.numpy())
    srt = torch.sort(z, dim=1, descending=True).values
    gap = (srt[:, 0] - srt[:, 1]).numpy()
    sel = gap > 0
    assert np.array_equal(arg[sel], zarg.numpy()[sel])
    assert np.array_equal(second, srt[:, 1].numpy())


def pin_epilogue_single_channel(orc):
    """C == 1 reduces to m * clamp(IN(m x), -1, 1)."""
    g = torch.Generator().manual_seed(4)
    x = torch.randn(2, 1, 50, generator=g).float()
    m = torch.tensor([-1.75], dtype=torch.float32)
    y, arg, second = orc.epilogue(x.numpy(), m.numpy(), EPS)
    ref = (-1.75 * torch.clamp(F.instance_norm(x.double() * -1.75, eps=EPS), -1, 1)).float()
    assert np.array_equal(y, ref[:, 0].numpy())
    assert np.all(arg == 0) and np.all(np.isneginf(second))


def pin_epilogue_clamp_saturation(orc):
    """An outlier normalises to sqrt(S-1) > 1 and clamps to exactly hi, so the
    channel contributes exactly m_c there; the other entries to exactly m_c*lo."""
    S = 17
    x = np.zeros((1, 2, S), dtype=np.float32)
    x[0, 0, 5] = 100.0                      # channel 0: one outlier
    x[0, 1, :] = np.arange(S, dtype=np.float32)
    m = np.array([0.75, -0.5], dtype=np.float32)
    y, arg, _ = orc.epilogue(x, m, EPS)
    # channel 0: IN = +4.0 at s=5 (clamps to 1 -> exactly 0.75), about -0.25 elsewhere
    assert y[0, 5] == np.float32(0.75) and arg[0, 5] == 0
    # channel 1 (m=-0.5): IN(-0.5*s) runs from +1.63 down to -1.63; at s=16 it
    # clamps to -1, giving exactly (-0.5)*(-1) = 0.5, the maximum there
    assert y[0, 16] == np.float32(0.5) and arg[0, 16] == 1
    # at s=0 channel 1 clamps to +1 (z = -0.5) and channel 0 wins with about -0.1875
    assert arg[0, 0] == 0 and abs(float(y[0, 0]) + 0.1875) < 1e-5


def pin_epilogue_hand_max(orc):
    """Two channels, two positions per slice, worked by hand: IN of a 2-value
    slice {p, q} is +-(|p-q|/2)/sqrt((p-q)^2/4 + eps)."""
    x = np.array([[[1.0, 3.0], [10.0, 2.0]]], dtype=np.float32)   # [N=1, C=2, S=2]
    m = np.array([2.0, 0.5], dtype=np.float32)
    y, arg, _ = orc.epilogue(x, m, EPS, -0.9, 0.9)
    # c=0: v = {2, 6}: t = {-r0, +r0} with r0 = 2/sqrt(4+eps) ~ 0.99999875 -> clamp +-0.9 -> z = {-1.8, 1.8}
    # c=1: v = {5, 1}: t = {+r1, -r1} with r1 = 2/sqrt(4+eps) -> clamp -> z = {0.45, -0.45}
    assert y[0, 0] == np.float32(0.45) and arg[0, 0] == 1
    assert y[0, 1] == np.float32(1.8) and arg[0, 1] == 0


def pin_epilogue_ties_lowest_index(orc):
    """Equal channels give equal z; the lowest channel index wins."""
    x = np.tile(np.arange(8, dtype=np.float32), (1, 3, 1))   # [1, 3, 8] identical slices
    m = np.array([1.0, 1.0, 1.0], dtype=np.float32)
    y, arg, second = orc.epilogue(x, m, EPS)
    assert np.all(arg == 0) and np.array_equal(second, y)


def pin_epilogue_page_shape(orc):
    """The page's shape rule: [N,16,14,30,30] reduces over C to [N,14,30,30]."""
    facts = read_facts()
    in_shape = tuple(int(v) for v in facts["epilogue_in_shape"].split(","))
    out_shape = tuple(int(v) for v in facts["epilogue_out_shape"].split(","))
    assert int(facts["epilogue_slice_len"]) == int(np.prod(in_shape[2:]))
    n = 2   # the first two samples; the rule does not depend on N
    g = torch.Generator().manual_seed(8)
    x = torch.randn((n,) + in_shape[1:], generator=g).float()
    m = torch.randn(in_shape[1], generator=g).float()
    y, arg, _ = orc.epilogue(x.numpy(), m.numpy(), EPS)
    assert y.shape == (n,) + out_shape[1:] and arg.shape == y.shape
    z = _epilogue_torch(x.double(), m.double()).float()
    assert np.array_equal(y, z.max(dim=1).values.numpy())


# ---------------------------------------------------------------------------
# BatchNorm (training)
# ---------------------------------------------------------------------------
def pin_batchnorm_vs_torch(orc):
    """torch's float64 batch_norm(training=True) with running stats, times the
    page's scale factor."""
    facts = read_facts()
    scale = float(facts["bn_scale"])
    momentum = float(facts["bn_momentum"])
    g = torch.Generator().manual_seed(13)
    x = (torch.randn(4, 6, 5, 7, generator=g) * 1.7 - 0.3).float()
    gamma = (1 + 0.1 * torch.randn(6, generator=g)).float()
    beta = (0.1 * torch.randn(6, generator=g)).float()
    rm = torch.linspace(-1, 1, 6, dtype=torch.float64)
    rv = torch.linspace(0.5, 2, 6, dtype=torch.float64)
    rm_t, rv_t = rm.clone(), rv.clone()
    ref = scale * F.batch_norm(x.double(), rm_t, rv_t, gamma.double(), beta.double(),
                               training=True, momentum=momentum, eps=EPS)
    y, rm_o, rv_o, mean, var = orc.batchnorm_train(x.numpy(), gamma.numpy(), beta.numpy(), scale,
                                                   rm.numpy(), rv.numpy(), momentum, EPS)
    assert np.max(np.abs(y - ref.float().numpy())) <= 1e-6
    assert np.max(np.abs(rm_o - rm_t.numpy())) <= 1e-14
    assert np.max(np.abs(rv_o - rv_t.numpy())) <= 1e-14


def pin_batchnorm_is_instancenorm_of_channel_view(orc):
    """Without affine terms, BN of channel c equals IN of all (n, s) values of
    channel c gathered into one slice."""
    g = torch.Generator().manual_seed(17)
    x = torch.randn(3, 4, 10, generator=g).float()
    y, _, _, mean, var = orc.batchnorm_train(x.numpy(), None, None, 1.0, None, None, 0.1, EPS)
    xc = x.permute(1, 0, 2).reshape(4, 30).contiguous().numpy()
    yi, mi, vi = orc.instancenorm(xc, EPS)
    assert np.array_equal(y.transpose(1, 0, 2).reshape(4, 30), yi)
    assert np.array_equal(mean, mi) and np.array_equal(var, vi)


def pin_batchnorm_running_stats_closed_form(orc):
    """From running_mean = 0 and running_var = 1 one step gives
    rm = 0.1*mu and rv = 0.9 + 0.1*var*n/(n-1) (unbiased estimator)."""
    x = np.array([[[1.0, 2.0]], [[3.0, 6.0]]], dtype=np.float32)   # N=2, C=1, S=2
    # channel values {1,2,3,6}: mu = 3, biased var = 7/2, unbiased = 14/3
    _, rm, rv, mean, var = orc.batchnorm_train(x, None, None, 1.0, [0.0], [1.0], 0.1, EPS)
    assert mean[0] == 3.0 and var[0] == 3.5
    assert abs(rm[0] - 0.3) <= 1e-16
    assert abs(rv[0] - (0.9 + 0.1 * 14.0 / 3.0)) <= 1e-15


def pin_batchnorm_affine_and_scale(orc):
    """y = scale*(gamma*xhat + beta): scale applies after beta."""
    x = np.array([[[1.0, 3.0]], [[1.0, 3.0]]], dtype=np.float32)   # channel {1,3,1,3}: xhat = -+r
    r = 1.0 / math.sqrt(1.0 + EPS)
    y, _, _, _, _ = orc.batchnorm_train(x, np.array([3.0], np.float32),
                                        np.array([0.5], np.float32), 2.0, None, None, 0.1, EPS)
    assert abs(float(y[0, 0, 0]) - 2.0 * (3.0 * -r + 0.5)) <= 4e-7
    assert abs(float(y[1, 0, 1]) - 2.0 * (3.0 * r + 0.5)) <= 4e-7


# ---------------------------------------------------------------------------
# InstanceNorm with per-channel affine parameters
# ---------------------------------------------------------------------------
def pin_instancenorm_affine_vs_torch(orc):
    """torch's float64 instance_norm with weight and bias (an independent
    library routine) on random slices of several channels and samples."""
    g = torch.Generator().manual_seed(41)
    x = torch.randn(3, 5, 4, 7, generator=g, dtype=torch.float64) * 2.0 + 0.7
    w = torch.randn(5, generator=g, dtype=torch.float64)
    b = torch.randn(5, generator=g, dtype=torch.float64)
    ref = F.instance_norm(x, weight=w, bias=b, eps=EPS)
    y, _, _ = orc.instancenorm_affine(x.numpy(), w.numpy(), b.numpy(), EPS)
    assert np.max(np.abs(y - ref.numpy())) <= 1e-13


def pin_instancenorm_affine_two_valued_closed_form(orc):
    """A slice alternating a, b has xhat = -+k, k = h/sqrt(h^2 + eps), h = |b-a|/2;
    channel c then maps it to gamma_c*(-+k) + beta_c, the same for every sample n."""
    N, C, S = 2, 3, 6
    a, bb = 1.0, 4.0
    x = np.tile(np.array([a, bb] * (S // 2)), (N, C, 1))
    gam = np.array([2.0, -0.5, 3.0])
    bet = np.array([0.25, 1.0, -2.0])
    h = abs(bb - a) / 2.0
    k = h / math.sqrt(h * h + EPS)
    y, mean, var = orc.instancenorm_affine(x, gam, bet, EPS)
    for n in range(N):
        for c in range(C):
            assert abs(y[n, c, 0] - (gam[c] * -k + bet[c])) <= 1e-15
            assert abs(y[n, c, 1] - (gam[c] * k + bet[c])) <= 1e-15
    assert np.all(mean == 2.5) and np.all(var == 2.25)


def pin_instancenorm_affine_defaults(orc):
    """gamma = beta = None is affine=False: the same values as InstanceNorm."""
    x = np.random.default_rng(43).standard_normal((2, 3, 11))
    y, _, _ = orc.instancenorm_affine(x, None, None, EPS)
    ref = F.instance_norm(torch.from_numpy(x), eps=EPS).numpy()
    assert np.max(np.abs(y - ref)) <= 1e-14


# ---------------------------------------------------------------------------
# BatchNorm in eval mode (running statistics), then the scale factor
# ---------------------------------------------------------------------------
def pin_batchnorm_eval_vs_torch(orc):
    """torch's float64 batch_norm with training=False (running statistics),
    times the scale factor."""
    g = torch.Generator().manual_seed(47)
    x = torch.randn(4, 6, 5, 3, generator=g, dtype=torch.float64) * 1.5 - 0.3
    rm = torch.randn(6, generator=g, dtype=torch.float64)
    rv = torch.rand(6, generator=g, dtype=torch.float64) * 3.0 + 0.1
    w = torch.randn(6, generator=g, dtype=torch.float64)
    b = torch.randn(6, generator=g, dtype=torch.float64)
    ref = 2.0 * F.batch_norm(x, rm, rv, weight=w, bias=b, training=False, eps=EPS)
    y = orc.batchnorm_eval(x.numpy(), w.numpy(), b.numpy(), 2.0, rm.numpy(), rv.numpy(), EPS)
    assert np.max(np.abs(y - ref.numpy())) <= 1e-13


def pin_batchnorm_eval_exact_values(orc):
    """Hand-computable values (eps chosen so that sqrt(rv + eps) is exact):
    rv = 3.75, eps = 0.25 -> sqrt = 2; gamma = 3, beta = 0.5, scale = 2,
    rm = 1: x = 5 -> 2*(3*4/2 + 0.5) = 13; x = -1 -> 2*(3*-1 + 0.5) = -5."""
    x = np.array([[[5.0, -1.0, 1.0]]])
    y = orc.batchnorm_eval(x, [3.0], [0.5], 2.0, [1.0], [3.75], 0.25)
    assert y.tolist() == [[[13.0, -5.0, 1.0]]]


def pin_batchnorm_eval_page_folding(orc):
    """Kimi-K2.6__l2_p73, block 2 folds eval BatchNorm and the scale into a
    per-channel factor gamma*s/sqrt(rv+eps) and a bias ((b - rm)*gamma/
    sqrt(rv+eps) + beta)*s of the preceding convolution; with an identity
    convolution (weight 1, bias 0) that is y = x*factor + bias_c."""
    rng = np.random.default_rng(53)
    N, C, S = 3, 4, 9
    x = rng.standard_normal((N, C, S)) * 3.0
    gam, bet = rng.standard_normal(C), rng.standard_normal(C)
    rm, rv = rng.standard_normal(C), rng.uniform(0.2, 2.0, C)
    s = 2.0
    factor = gam * s / np.sqrt(rv + EPS)
    bias = ((0.0 - rm) * gam / np.sqrt(rv + EPS) + bet) * s
    y = orc.batchnorm_eval(x, gam, bet, s, rm, rv, EPS)
    assert np.max(np.abs(y - (x * factor[None, :, None] + bias[None, :, None]))) <= 1e-12


def pin_batchnorm_eval_equals_train_with_batch_stats(orc):
    """With the running statistics set to the batch mean and the biased batch
    variance, the eval form gives the training form's output."""
    rng = np.random.default_rng(59)
    x = (rng.standard_normal((5, 3, 8)) * 2.0 + 1.0).astype(np.float32)
    gam = rng.standard_normal(3).astype(np.float32)
    bet = rng.standard_normal(3).astype(np.float32)
    yt, _, _, mean, var = orc.batchnorm_train(x, gam, bet, 2.0, None, None, 0.1, EPS)
    ye = orc.batchnorm_eval(x, gam, bet, 2.0, mean, var, EPS)
    assert np.array_equal(ye.astype(np.float32), yt)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
