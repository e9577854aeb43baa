"""fnorm_batchnorm_train_noalloc: the BatchNorm entry point for callers that
cannot allocate device memory (fixed memory budgets, plugins whose host owns
the allocator, loops where a synchronising cudaMalloc is not allowed). It
uses the library's own static device scratch instead of a caller workspace.

Its results must match fnorm_batchnorm_train's within the parity tolerance,
on two calls in a row (the second call finds the scratch holding the first
call's partials). This file is collected last so that a run stopping at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import normalization_reduction_gb300 as fn
from normalization_reduction_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = 1e-4   # max-abs, as in the other fp32 parity tests
SCRATCH_BYTES = 2 << 20


def _with_workspace(x, g, b, rm, rv):
    N, C = x.shape[0], x.shape[1]
    S = x[0, 0].numel()
    y = torch.empty_like(x)
    ws = torch.empty(fn.fnorm_batchnorm_workspace_size(N, C, S), dtype=torch.uint8,
                     device=x.device)
    sm, sr = torch.empty(C, device=x.device), torch.empty(C, device=x.device)
    fn.fnorm_batchnorm_train(x, y, g, b, 2.0, rm, rv, 0.1, 1e-5, sm, sr, N, C, S, ws, ws.numel())
    return y, sm, sr


def _no_alloc(x, g, b, rm, rv):
    N, C = x.shape[0], x.shape[1]
    S = x[0, 0].numel()
    y = torch.empty_like(x)
    sm, sr = torch.empty(C, device=x.device), torch.empty(C, device=x.device)
    fn.fnorm_batchnorm_train_noalloc(x, y, g, b, 2.0, rm, rv, 0.1, 1e-5, sm, sr, N, C, S)
    return y, sm, sr


@pytest.mark.parametrize("shapes", [[(8, 64, 126, 126), (4, 6, 1000)]])
def test_no_alloc_matches_workspace_entry_point(shapes):
    dev = torch.device("cuda", torch.cuda.current_device())
    for i, shape in enumerate(shapes):          # two calls in a row
        x, g, b, rm, rv = inputs.batchnorm(dev, shape=shape, seed=500 + i)
        rm_a, rv_a, rm_b, rv_b = rm.clone(), rv.clone(), rm.clone(), rv.clone()
        y_a, sm_a, sr_a = _with_workspace(x, g, b, rm_a, rv_a)
        y_b, sm_b, sr_b = _no_alloc(x, g, b, rm_b, rv_b)
        torch.cuda.synchronize()
        for a, b_ in ((y_a, y_b), (sm_a, sm_b), (sr_a, sr_b), (rm_a, rm_b), (rv_a, rv_b)):
            assert float((a - b_).abs().max()) <= TOL


def test_no_alloc_rejects_shapes_beyond_the_scratch():
    dev = torch.device("cuda", torch.cuda.current_device())
    N, C, S = 4096, 64, 4          # partials need 4096*64*16 bytes > 2 MiB
    assert fn.fnorm_batchnorm_workspace_size(N, C, S) > SCRATCH_BYTES
    x = torch.zeros(1, device=dev)
    with pytest.raises(fn.FnormError) as e:
        fn.fnorm_batchnorm_train_noalloc(x, x, None, None, 1.0, None, None, 0.1, 1e-5, None,
                                         None, N, C, S)
    assert e.value.status == fn.Status.ERR_UNSUPPORTED
