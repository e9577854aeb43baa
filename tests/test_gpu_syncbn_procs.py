"""Synchronised training BatchNorm as real processes through the library: R
processes (gloo process group, all on GPU 0) each call
syncbn.sync_batch_norm_train on their shard of the batch --
fnorm_batchnorm_local_stats, the all-gather of the [C][4] statistics over
gloo, then fnorm_batchnorm_apply_stats. The concatenated outputs and every
rank's running statistics must equal the oracle's BatchNorm of the whole
batch (page Kimi-K2.6__l2_p73, block 1: statistics over (N, H, W)). One case
gives a rank an empty shard, one runs the library calls on a stream other
than torch's current one.

The processes do not wait on one another inside any kernel: the only exchange
is the host-side gloo all-gather between the two library calls."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as tdist
import torch.multiprocessing as mp

from normalization_reduction_gb300 import inputs
from tests.gpu_util import assert_close

pytestmark = pytest.mark.gpu

EPS, MOM, SCALE = 1e-5, 0.1, 2.0


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shape(splits, C, spatial):
    return (sum(splits), C) + tuple(spatial)


def _worker(rank, size, port, outdir, splits, C, spatial, side_stream, seed):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=size)
    torch.cuda.set_device(0)
    from normalization_reduction_gb300 import syncbn
    x, g, b, rm, rv = inputs.batchnorm("cuda", shape=_shape(splits, C, spatial), seed=seed)
    lo = sum(splits[:rank])
    shard = x[lo:lo + splits[rank]].contiguous()
    s = torch.cuda.Stream() if side_stream else None
    y = syncbn.sync_batch_norm_train(shard, g, b, rm, rv, MOM, EPS, SCALE, stream=s)
    if s is not None:
        torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    np.save(os.path.join(outdir, f"y_{rank}.npy"), y.cpu().numpy())
    np.save(os.path.join(outdir, f"rm_{rank}.npy"), rm.cpu().numpy())
    np.save(os.path.join(outdir, f"rv_{rank}.npy"), rv.cpu().numpy())
    tdist.barrier()
    tdist.destroy_process_group()


@pytest.mark.parametrize("splits,C,spatial,side_stream", [
    ([3, 5], 64, (32, 32), False),
    ([3, 0, 5], 16, (9, 11), True),
    ([4, 4], 8, (3, 5), True),        # runs of 15 values: the column forms
], ids=["2ranks", "3ranks_empty_side_stream", "2ranks_columns_side_stream"])
def test_processes_match_whole_batch(orc, tmp_path, splits, C, spatial, side_stream):
    seed = 4242 + len(splits)
    size = len(splits)
    mp.spawn(_worker, args=(size, _free_port(), str(tmp_path), splits, C, spatial, side_stream,
                            seed), nprocs=size, join=True)
    shape = _shape(splits, C, spatial)
    x, g, b, rm, rv = inputs.batchnorm("cuda", shape=shape, seed=seed)
    S = int(np.prod(spatial))
    ref, rmo, rvo, _, _ = orc.batchnorm_train(x.cpu().numpy().reshape(shape[0], C, S),
                                              g.cpu().numpy(), b.cpu().numpy(), SCALE,
                                              rm.cpu().numpy(), rv.cpu().numpy(), MOM, EPS)
    ys = [np.load(tmp_path / f"y_{r}.npy") for r in range(size)]
    for r, n in enumerate(splits):
        assert ys[r].shape == (n, C) + tuple(spatial)
    got = np.concatenate(ys).reshape(ref.shape)
    assert_close(got, ref, torch.float32, f"{size} processes, splits {splits}")
    for r in range(size):
        assert np.max(np.abs(np.load(tmp_path / f"rm_{r}.npy") - rmo)) <= 1e-6
        assert np.max(np.abs(np.load(tmp_path / f"rv_{r}.npy") - rvo)) <= 2e-6
    # every rank merged the same gathered statistics in rank order
    rm0 = np.load(tmp_path / "rm_0.npy")
    assert all(np.array_equal(np.load(tmp_path / f"rm_{r}.npy"), rm0) for r in range(size))
