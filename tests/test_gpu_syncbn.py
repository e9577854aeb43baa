"""Multi-process BatchNorm's GPU side, with the ranks emulated on one GPU:
the batch is split along N into shards, each shard's statistics come from
fnorm_batchnorm_local_stats, the stacked [R][C][4] array (what an all-gather
produces) feeds fnorm_batchnorm_apply_stats for every shard, and the
concatenated outputs and every shard's running statistics match the oracle's
BatchNorm of the whole batch."""
import numpy as np
import pytest
import torch

import normalization_reduction_gb300 as fn
from normalization_reduction_gb300 import inputs, syncbn
from tests.gpu_util import assert_close, dev

pytestmark = pytest.mark.gpu

EPS, MOM, SCALE = 1e-5, 0.1, 2.0


def local_stats(shard):
    N, C = shard.shape[0], shard.shape[1]
    S = int(np.prod(shard.shape[2:]))
    out = torch.empty((C, 4), device=dev())
    nb = max(fn.fnorm_batchnorm_workspace_size(N, C, S), 1)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev())
    fn.fnorm_batchnorm_local_stats(shard, out, N, C, S, ws, nb)
    return out


@pytest.mark.parametrize("splits", [[2, 2], [3, 5], [4, 0, 3], [1, 1, 1, 1, 4]])
@pytest.mark.parametrize("spatial", [(9, 11), (1,), (3,), (4, 4)],
                         ids=["S99", "S1", "S3", "S16"])
def test_emulated_ranks_match_whole_batch(orc, splits, spatial):
    """Runs of more than 16 values take the per-unit kernels, shorter runs the
    column kernels (column statistics; rank-ordered fold per column)."""
    shape = (sum(splits) * (64 if len(spatial) == 1 else 1), 6) + spatial
    splits = [n * (64 if len(spatial) == 1 else 1) for n in splits]
    x, g, b, rm, rv = inputs.batchnorm(dev(), shape=shape, seed=55 + len(splits))
    C = shape[1]
    S = int(np.prod(spatial))
    shards, lo = [], 0
    for n in splits:
        shards.append(x[lo:lo + n].contiguous())
        lo += n
    stats_all = torch.stack([local_stats(s) for s in shards]).contiguous()
    outs, rms, rvs = [], [], []
    for s in shards:
        y = torch.empty_like(s)
        rm_r, rv_r = rm.clone(), rv.clone()
        fn.fnorm_batchnorm_apply_stats(s, y, stats_all, len(splits), g, b, SCALE, rm_r, rv_r, MOM,
                                       EPS, None, None, s.shape[0], C, S)
        outs.append(y)
        rms.append(rm_r)
        rvs.append(rv_r)
    torch.cuda.synchronize()
    ref, rmo, rvo, mean, var = orc.batchnorm_train(x.cpu().numpy().reshape(shape[0], C, S),
                                                   g.cpu().numpy(), b.cpu().numpy(), SCALE,
                                                   rm.cpu().numpy(), rv.cpu().numpy(), MOM, EPS)
    got = torch.cat(outs).cpu().numpy().reshape(ref.shape)
    assert_close(got, ref, torch.float32, f"splits {splits} spatial {spatial}")
    for rm_r, rv_r in zip(rms, rvs):
        assert np.max(np.abs(rm_r.cpu().numpy() - rmo)) <= 1e-6
        assert np.max(np.abs(rv_r.cpu().numpy() - rvo)) <= 2e-6
    sa = stats_all.cpu().numpy()
    assert np.array_equal(sa[:, :, 0].sum(axis=0), np.full(C, shape[0] * S, dtype=np.float32))


def test_single_process_helper_equals_train(orc):
    x, g, b, rm, rv = inputs.batchnorm(dev(), shape=(4, 8, 30, 30), seed=8)
    rm2, rv2 = rm.clone(), rv.clone()
    y = syncbn.sync_batch_norm_train(x, g, b, rm, rv, MOM, EPS, SCALE)
    y2 = fn.batch_norm_train(x, g, b, rm2, rv2, MOM, EPS, SCALE)
    torch.cuda.synchronize()
    assert float((y - y2).abs().max()) <= 1e-5
    assert float((rm - rm2).abs().max()) <= 1e-6 and float((rv - rv2).abs().max()) <= 1e-6


def test_empty_shard_stats_are_identity():
    x = torch.empty((0, 5, 7), device=dev())
    out = torch.full((5, 4), 7.0, device=dev())
    fn.fnorm_batchnorm_local_stats(x, out, 0, 5, 7, None, 0)
    torch.cuda.synchronize()
    assert bool((out == 0).all())


def test_single_process_on_a_side_stream(orc):
    """The library calls on a stream other than torch's current one: the
    inputs are written on the current stream just before the call, and the
    result equals the oracle once the side stream is synchronised."""
    x, g, b, rm, rv = inputs.batchnorm(dev(), shape=(6, 8, 20, 20), seed=9)
    x2 = torch.empty_like(x)
    side = torch.cuda.Stream()
    rm0, rv0 = rm.cpu().numpy(), rv.cpu().numpy()
    for _ in range(3):
        x2.copy_(x)                     # on the current stream
        rm.copy_(torch.from_numpy(rm0).to(dev()))
        rv.copy_(torch.from_numpy(rv0).to(dev()))
        y = syncbn.sync_batch_norm_train(x2, g, b, rm, rv, MOM, EPS, SCALE, stream=side)
        x2.fill_(1e30)                  # the next step's writes, ordered after the call
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        ref, rmo, rvo, _, _ = orc.batchnorm_train(x.cpu().numpy().reshape(6, 8, 400),
                                                  g.cpu().numpy(), b.cpu().numpy(), SCALE,
                                                  rm0, rv0, MOM, EPS)
        assert_close(y.cpu().numpy().reshape(6, 8, 400), ref, torch.float32, "side stream")
        assert np.max(np.abs(rm.cpu().numpy() - rmo)) <= 1e-6
