"""Repetition under load: every kernel family is launched many times,
alternating between two streams, and every result must equal the first one
bit for bit, with no error recorded. A race in
a cluster exchange or an mbarrier protocol shows up here as a rare mismatch or
a timeout."""
import os

import pytest
import torch

import normalization_reduction_gb300 as fn
from normalization_reduction_gb300 import inputs
from tests.gpu_util import dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

EPS = 1e-5
REPEATS = int(os.environ.get("FNORM_STRESS_REPEATS", "40"))


def _cases():
    cases = []
    for k, (shape, dt) in enumerate((((16, 64, 512, 512), torch.float32),      # split, 8-CTA clusters
                                     ((8, 8, 1024, 1024), torch.bfloat16),     # split, 16-CTA clusters
                                     ((256, 64, 16, 16), torch.bfloat16),      # group kernel
                                     ((1, 3, 2048, 2048), torch.float32))):    # stream, few slices
        x = inputs.normal(shape, 800 + k, dev()).to(dt)
        N, C = shape[0], shape[1]
        S = shape[2] * shape[3]
        c = fn.FNORM_F32 if dt == torch.float32 else fn.FNORM_BF16

        def run(st, x=x, N=N, C=C, S=S, c=c):
            y = torch.empty_like(x)
            fn.fnorm_instancenorm(x, y, N, C, S, c, c, EPS, None, None, st)
            return [y]
        cases.append(run)
    xe, m = inputs.epilogue(dev())

    def run_epi(st):
        y = torch.empty((128, 12600), device=dev())
        a = torch.empty((128, 12600), dtype=torch.int64, device=dev())
        fn.fnorm_instancenorm_epilogue(xe, m, y, a, 128, 16, 12600, EPS, -1.0, 1.0, st)
        return [y, a]
    cases.append(run_epi)
    xb, g, b, _, _ = inputs.batchnorm(dev(), shape=(32, 64, 126, 126))
    ws = torch.empty(fn.fnorm_batchnorm_workspace_size(32, 64, 126 * 126), dtype=torch.uint8,
                     device=dev())

    def run_bn(st):
        y = torch.empty_like(xb)
        sm = torch.empty(64, device=dev())
        fn.fnorm_batchnorm_train(xb, y, g, b, 2.0, None, None, 0.1, EPS, sm, None, 32, 64,
                                 126 * 126, ws, ws.numel(), st)
        return [y, sm]
    cases.append(run_bn)
    return cases


@pytest.mark.parametrize("case", range(6))
def test_repeated_launches_are_identical(case):
    run = _cases()[case]
    st = torch.cuda.current_stream()
    first = run(st)
    torch.cuda.synchronize()
    s2 = torch.cuda.Stream()
    for i in range(REPEATS):
        with torch.cuda.stream(s2 if i % 2 else st):
            outs = run(s2 if i % 2 else st)
        torch.cuda.synchronize()
        for a, b in zip(first, outs):
            assert torch.equal(a, b), f"repeat {i}"
    assert fn.fnorm_get_last_error() == fn.Status.OK
