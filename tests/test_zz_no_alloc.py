"""fnorm_batchnorm_train_noalloc: the BatchNorm entry point for callers that
cannot allocate device memory (fixed memory budgets, plugins whose host owns
the allocator, loops where a synchronising cudaMalloc is not allowed). It
uses the library's own static device scratch instead of a caller workspace.

Both entry points run the same kernels on the same partial-statistics layout,
so the results must be bit-identical, call after call: a small shape, then a
large one, then a shape of runs of at most 16 values (the column form, which
keeps its coefficients at another offset of the scratch), then the small one
again -- so that later calls read scratch regions that earlier calls left
holding other partials. This file is collected last so that a run stopping at
the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import normalization_reduction_gb300 as fn
from normalization_reduction_gb300 import inputs

pytestmark = pytest.mark.gpu

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


@pytest.mark.parametrize("shapes", [[(4, 6, 1000), (8, 64, 126, 126), (64, 8, 4),
                                     (4, 6, 1000)]])
def test_no_alloc_matches_workspace_entry_point(shapes):
    dev = torch.device("cuda", torch.cuda.current_device())
    for i, shape in enumerate(shapes):          # calls in a row on the shared scratch
        x, g, b, rm, rv = inputs.batchnorm(dev, shape=shape, seed=500 + i)
        rm_a, rv_a, rm_b, rv_b = rm.clone(), rv.clone(), rm.clone(), rv.clone()
        y_a, sm_a, sr_a = _with_workspace(x, g, b, rm_a, rv_a)
        y_b, sm_b, sr_b = _no_alloc(x, g, b, rm_b, rv_b)
        torch.cuda.synchronize()
        for a, b_ in ((y_a, y_b), (sm_a, sm_b), (sr_a, sr_b), (rm_a, rm_b), (rv_a, rv_b)):
            assert torch.equal(a, b_), shape


def test_no_alloc_validates_like_the_workspace_entry_point():
    """Argument errors are those of fnorm_batchnorm_train even for shapes too
    large for the scratch (the size check comes after the validation)."""
    N, C, S = 4096, 64, 4
    assert fn.fnorm_batchnorm_workspace_size(N, C, S) > SCRATCH_BYTES
    fake = 1 << 40   # never dereferenced: every call below fails validation first
    cases = [dict(eps=-1.0), dict(y=None), dict(x=fake + 2)]
    for kw in cases:
        a = dict(x=fake, y=fake + (1 << 32), eps=1e-5)
        a.update(kw)
        with pytest.raises(fn.FnormError) as e1:
            fn.fnorm_batchnorm_train_noalloc(a["x"], a["y"], None, None, 1.0, None, None, 0.1,
                                             a["eps"], None, None, N, C, S)
        with pytest.raises(fn.FnormError) as e2:
            fn.fnorm_batchnorm_train(a["x"], a["y"], None, None, 1.0, None, None, 0.1, a["eps"],
                                     None, None, N, C, S, fake + (1 << 36), 1 << 30)
        assert e1.value.status == e2.value.status != fn.Status.ERR_UNSUPPORTED, kw


def test_no_alloc_rejects_shapes_beyond_the_scratch():
    dev = torch.device("cuda", torch.cuda.current_device())
    N, C, S = 4096, 64, 4          # partials need 4096*64*16 bytes > 2 MiB
    assert fn.fnorm_batchnorm_workspace_size(N, C, S) > SCRATCH_BYTES
    x = torch.zeros(1, device=dev)
    with pytest.raises(fn.FnormError) as e:
        fn.fnorm_batchnorm_train_noalloc(x, x, None, None, 1.0, None, None, 0.1, 1e-5, None,
                                         None, N, C, S)
    assert e.value.status == fn.Status.ERR_UNSUPPORTED
