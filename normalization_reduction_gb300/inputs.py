"""Seeded synthetic inputs with the shapes and value distributions of the
pages' workloads. This module holds no arithmetic of the method itself; the
CUDA path and the oracle both take their inputs from here.

Workloads (all NCHW / NCDHW contiguous, fp32 unless stated):

* ``instancenorm_small``   x[2,4,16,16] ~ N(0,1), slice (n=1,c=3) set to 5.0.
* ``instancenorm_large``   x[112,64,512,512] ~ N(0,1) -- the InstanceNorm2d(64)
  input of the page Kimi-K2.6__l1_p34 (7168 slices of 512x512).
* ``epilogue``             x[128,16,14,30,30], channel c ~ N(mu_c, s_c) with
  mu_c ~ U(-0.5,0.5), s_c ~ U(0.2,2); m[16] ~ N(0,1) -- the Conv3d output and
  multiplier of the page Kimi-K2.6__l2_p79 (conv replaced by generated data).
* ``batchnorm``            x[128,64,126,126] per-channel as above;
  gamma = 1 + 0.1 N(0,1), beta = 0.1 N(0,1), running_mean = 0, running_var = 1
  -- the Conv2d output of the page Kimi-K2.6__l2_p73.
* ``instancenorm_affine``  x as ``instancenorm_large`` (seed 1006) with
  per-channel gamma = 1 + 0.1 N(0,1), beta = 0.1 N(0,1) -- InstanceNorm2d(64)
  with its affine=True option.
* ``batchnorm_eval``       x as ``batchnorm`` (seed 1007) with gamma/beta as
  there and running statistics of a model that has seen such data:
  running_mean = mu_c + 0.05 N(0,1), running_var = s_c^2 * U(0.8, 1.2).
* ``instancenorm_sweep``   bf16 x ~ N(3,2) (rounded from fp32), N = 8,
  2^30 elements in total, slice length S from 256 to 1,048,576.

Random numbers come from torch generators seeded per workload; large tensors
are drawn on the device they are requested on. Parameters that are drawn per
channel always come from a CPU generator so that they do not depend on the
device.
"""
from __future__ import annotations

import torch

SEED_SMALL = 1001
SEED_LARGE = 1002
SEED_EPILOGUE = 1003
SEED_BATCHNORM = 1004
SEED_SWEEP = 1005
SEED_AFFINE = 1006
SEED_BN_EVAL = 1007

SHAPE_SMALL = (2, 4, 16, 16)
SHAPE_LARGE = (112, 64, 512, 512)
SHAPE_EPILOGUE = (128, 16, 14, 30, 30)
SHAPE_BATCHNORM = (128, 64, 126, 126)
SWEEP_TOTAL = 1 << 30
SWEEP_N = 8
SWEEP_S = tuple(4 ** k for k in range(4, 11))  # 256 ... 1,048,576


def _gen(seed: int, device) -> torch.Generator:
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    return g


def normal(shape, seed: int, device="cpu", mean: float = 0.0, std: float = 1.0,
           dtype=torch.float32) -> torch.Tensor:
    """x ~ N(mean, std) drawn in fp32 on ``device`` then cast to ``dtype``."""
    g = _gen(seed, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x if dtype == torch.float32 else x.to(dtype)


def uniform(shape, seed: int, device="cpu", lo: float = 0.0, hi: float = 1.0) -> torch.Tensor:
    g = _gen(seed, device)
    x = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
    return x.mul_(hi - lo).add_(lo)


def per_channel_normal(shape, seed: int, device="cpu"):
    """x[:, c] ~ N(mu_c, s_c), mu_c ~ U(-0.5, 0.5), s_c ~ U(0.2, 2).

    Returns (x, mu, s) with mu/s the per-channel draws (CPU float32).
    """
    C = shape[1]
    gc = _gen(seed, "cpu")
    mu = torch.rand(C, generator=gc) - 0.5
    s = torch.rand(C, generator=gc) * 1.8 + 0.2
    x = normal(shape, seed + 100_000, device)
    bshape = (1, C) + (1,) * (len(shape) - 2)
    x.mul_(s.to(device).view(bshape)).add_(mu.to(device).view(bshape))
    return x, mu, s


def instancenorm_small(device="cpu") -> torch.Tensor:
    x = normal(SHAPE_SMALL, SEED_SMALL, device)
    x[1, 3].fill_(5.0)
    return x


def instancenorm_large(device="cuda", shape=SHAPE_LARGE, seed: int = SEED_LARGE) -> torch.Tensor:
    return normal(shape, seed, device)


def epilogue(device="cuda", shape=SHAPE_EPILOGUE, seed: int = SEED_EPILOGUE):
    """Returns (x [N,C,D,H,W], m [C]) on ``device``."""
    x, _, _ = per_channel_normal(shape, seed, device)
    gm = _gen(seed + 200_000, "cpu")
    m = torch.randn(shape[1], generator=gm)
    return x, m.to(device)


def batchnorm(device="cuda", shape=SHAPE_BATCHNORM, seed: int = SEED_BATCHNORM):
    """Returns (x, gamma, beta, running_mean, running_var) on ``device``."""
    x, _, _ = per_channel_normal(shape, seed, device)
    C = shape[1]
    gp = _gen(seed + 300_000, "cpu")
    gamma = 1.0 + 0.1 * torch.randn(C, generator=gp)
    beta = 0.1 * torch.randn(C, generator=gp)
    rm = torch.zeros(C)
    rv = torch.ones(C)
    return x, gamma.to(device), beta.to(device), rm.to(device), rv.to(device)


def sweep_shape(S: int, total: int = SWEEP_TOTAL, N: int = SWEEP_N):
    """[N, C, S] with N*C*S == total."""
    if total % (N * S):
        raise ValueError("total must be a multiple of N*S")
    return (N, total // (N * S), S)


def instancenorm_sweep(S: int, device="cuda", total: int = SWEEP_TOTAL, N: int = SWEEP_N,
                       seed: int | None = None) -> torch.Tensor:
    """bf16 x[N, C, S] ~ N(3, 2), rounded to nearest-even from fp32."""
    k = SWEEP_S.index(S) if (seed is None and S in SWEEP_S) else 0
    return normal(sweep_shape(S, total, N), SEED_SWEEP + k if seed is None else seed, device,
                  mean=3.0, std=2.0, dtype=torch.bfloat16)


def channel_affine(C: int, seed: int, device="cpu"):
    """gamma = 1 + 0.1 N(0,1), beta = 0.1 N(0,1), drawn per channel on the CPU."""
    gp = _gen(seed + 300_000, "cpu")
    gamma = 1.0 + 0.1 * torch.randn(C, generator=gp)
    beta = 0.1 * torch.randn(C, generator=gp)
    return gamma.to(device), beta.to(device)


def instancenorm_affine(device="cuda", shape=SHAPE_LARGE, seed: int = SEED_AFFINE):
    """Returns (x, gamma [C], beta [C]) on ``device``."""
    x = normal(shape, seed, device)
    gamma, beta = channel_affine(shape[1], seed, device)
    return x, gamma, beta


def batchnorm_eval(device="cuda", shape=SHAPE_BATCHNORM, seed: int = SEED_BN_EVAL):
    """Returns (x, gamma, beta, running_mean, running_var) on ``device``."""
    x, mu, s = per_channel_normal(shape, seed, device)
    C = shape[1]
    gamma, beta = channel_affine(C, seed, "cpu")
    gr = _gen(seed + 400_000, "cpu")
    rm = mu + 0.05 * torch.randn(C, generator=gr)
    rv = s * s * (0.8 + 0.4 * torch.rand(C, generator=gr))
    return x, gamma.to(device), beta.to(device), rm.to(device), rv.to(device)
