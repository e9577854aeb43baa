"""Concurrent use: several host threads, each on its own CUDA stream, call
different entry points at the same time (run alone, this includes their first
calls, so that plan selection and the once-per-device set-up race). Every
result must equal the one a sequential call gives, bit for bit, and no error
may be recorded."""
import threading

import pytest
import torch

import normalization_reduction_gb300 as fn
from normalization_reduction_gb300 import inputs
from tests.gpu_util import dev

pytestmark = pytest.mark.gpu

EPS = 1e-5


def _jobs():
    jobs = []
    # InstanceNorm on several kernel paths, both dtypes, affine and not
    for k, (S, dt) in enumerate(((256, torch.bfloat16), (3000, torch.float32),
                                 (65536, torch.float32), (262144, torch.bfloat16))):
        x = inputs.normal((2, 6, S), 700 + k, dev()).to(dt)
        g, b = inputs.channel_affine(6, 710 + k, dev())
        c = fn.FNORM_F32 if dt == torch.float32 else fn.FNORM_BF16

        def run(st, x=x, g=g, b=b, S=S, c=c, aff=k % 2 == 0):
            y = torch.empty_like(x)
            fn.fnorm_instancenorm_affine(x, y, g if aff else None, b if aff else None, 2, 6, S, c,
                                         c, EPS, None, None, st)
            return [y]
        jobs.append(run)
    # the epilogue
    xe, m = inputs.epilogue(dev(), shape=(6, 16, 14, 30, 30))

    def run_epi(st):
        y = torch.empty((6, 12600), device=dev())
        a = torch.empty((6, 12600), dtype=torch.int64, device=dev())
        fn.fnorm_instancenorm_epilogue(xe, m, y, a, 6, 16, 12600, EPS, -1.0, 1.0, st)
        return [y, a]
    jobs.append(run_epi)
    # BatchNorm train (own workspace and running statistics per call) and eval
    xb, gb, bb, _, _ = inputs.batchnorm(dev(), shape=(8, 12, 50, 50))

    def run_bn(st):
        y = torch.empty_like(xb)
        rm = torch.zeros(12, device=dev())
        rv = torch.ones(12, device=dev())
        ws = torch.empty(fn.fnorm_batchnorm_workspace_size(8, 12, 2500), dtype=torch.uint8,
                         device=dev())
        fn.fnorm_batchnorm_train(xb, y, gb, bb, 2.0, rm, rv, 0.1, EPS, None, None, 8, 12, 2500, ws,
                                 ws.numel(), st)
        return [y, rm, rv]
    jobs.append(run_bn)

    def run_eval(st):
        y = torch.empty_like(xb)
        rm = torch.linspace(-0.2, 0.2, 12, device=dev())
        rv = torch.linspace(0.5, 1.5, 12, device=dev())
        fn.fnorm_batchnorm_eval(xb, y, gb, bb, 2.0, rm, rv, EPS, 8, 12, 2500, st)
        return [y]
    jobs.append(run_eval)
    return jobs


def test_threads_and_streams_match_sequential():
    jobs = _jobs()
    torch.cuda.synchronize()
    results = [None] * len(jobs)
    errors = []

    def worker(i):
        try:
            s = torch.cuda.Stream()
            outs = []
            with torch.cuda.stream(s):
                for _ in range(5):
                    outs = jobs[i](s)
            s.synchronize()
            results[i] = outs
        except Exception as e:  # reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(jobs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    assert fn.fnorm_get_last_error() == fn.Status.OK
    st = torch.cuda.current_stream()
    for i, job in enumerate(jobs):
        ref = job(st)
        torch.cuda.synchronize()
        for a, b in zip(results[i], ref):
            assert torch.equal(a, b), f"job {i}"
