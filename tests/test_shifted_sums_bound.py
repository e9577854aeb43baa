"""Host-side model of the shifted one-pass statistics that the epilogue kernel
and the bf16 InstanceNorm kernel (slices over 16-CTA clusters) use per thread:
with K the thread's first value, d = fl(x - K), S = sum d, Q = sum d^2 (fused
multiply-add), all in fp32, then mean = K + S/n and M2 = Q - S^2/n. The
kernels' plans cap a thread's count at 160 values.

Because K is one of the values, (K - mean)^2 <= M2, so Q = M2 + n (K - mean)^2
<= (n + 1) M2. Recursive summation gives |err Q| <= g(n+2) Q and
|err S^2/n| <= 2 g(n) Q with g(k) = k u / (1 - k u), u = 2^-24, hence

    |M2_fp32 - M2| <= 3 (n + 1) g(n + 2) M2.

The model uses one accumulator; the kernels use four, which only shortens
each sum. The tests check the bound on the worst placement (an outlier as
K, values far from zero) and that a shift that is not one of the values
breaks it, so the bound depends on that property."""
import numpy as np
import pytest

U = 2.0 ** -24


def gamma(k):
    return k * U / (1.0 - k * U)


def shifted_one_pass(x, K=None):
    x = x.astype(np.float32)
    K = np.float32(x[0] if K is None else K)
    s = np.float32(0.0)
    q = np.float32(0.0)
    for v in x:
        d = np.float32(v - K)
        s = np.float32(s + d)
        q = np.float32(np.float64(d) * np.float64(d) + np.float64(q))   # one rounding, as the FMA
    n = np.float32(len(x))
    mean = np.float32(K + np.float32(s / n))
    m2 = max(np.float32(q - np.float32(s * np.float32(s / n))), np.float32(0.0))
    return float(mean), float(m2)


def exact_m2(x):
    x = x.astype(np.float64)
    return float(np.sum((x - x.mean()) ** 2))


@pytest.mark.parametrize("n", [4, 32, 100, 128, 160])
def test_bound_with_outlier_shift(n):
    rng = np.random.default_rng(1700 + n)
    bound = 3 * (n + 1) * gamma(n + 2)
    worst = 0.0
    for trial in range(60):
        x = (rng.standard_normal(n) * rng.uniform(0.01, 2.0) + rng.uniform(-1e3, 1e3)).astype(np.float32)
        if trial % 2 == 0:   # the worst placement: an outlier at the shift
            x[0] = np.float32(x[0] + rng.choice([-1.0, 1.0]) * rng.uniform(10.0, 1e3) * np.std(x))
        m2 = exact_m2(x)
        _, got = shifted_one_pass(x)
        worst = max(worst, abs(got - m2) / m2)
    assert worst <= bound, (n, worst, bound)


def test_constant_values_give_zero_and_exact_mean():
    x = np.full(160, 123.456, dtype=np.float32)
    mean, m2 = shifted_one_pass(x)
    assert m2 == 0.0 and mean == float(x[0])


def test_shift_outside_the_values_breaks_the_bound():
    """The bound needs K to be one of the values: shifting by 0 instead, on
    values near 1000 with unit spread, loses most of M2 to cancellation."""
    rng = np.random.default_rng(1799)
    n = 128
    x = (rng.standard_normal(n) + 1000.0).astype(np.float32)
    m2 = exact_m2(x)
    _, got = shifted_one_pass(x, K=0.0)
    assert abs(got - m2) / m2 > 3 * (n + 1) * gamma(n + 2)
    _, good = shifted_one_pass(x)
    assert abs(good - m2) / m2 <= 3 * (n + 1) * gamma(n + 2)
