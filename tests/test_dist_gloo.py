"""The multi-process host path on the CPU: two gloo ranks shard an
InstanceNorm and an epilogue workload by slice / sample with no data-path
collective, and the union of their results equals the single-process result;
the timing reduction returns the maximum over ranks."""
import os
import socket

import numpy as np
import torch
import torch.distributed as tdist
import torch.multiprocessing as mp

from normalization_reduction_gb300 import dist, inputs


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, size, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=size)
    import oracle
    orc = oracle.get()
    # InstanceNorm: shard the N*C slices of a small workload of the large shape family
    x = inputs.instancenorm_large("cpu", shape=(3, 5, 16, 16), seed=77).reshape(15, 256).numpy()
    lo, hi = dist.shard(15, rank, size)
    y, _, _ = orc.instancenorm(x[lo:hi])
    np.save(os.path.join(outdir, f"in_{rank}.npy"), y)
    # epilogue: shard the samples
    xe, m = inputs.epilogue("cpu", shape=(5, 4, 2, 3, 4), seed=78)
    lo, hi = dist.shard(5, rank, size)
    ye, _, _ = orc.epilogue(xe.numpy()[lo:hi], m.numpy())
    np.save(os.path.join(outdir, f"epi_{rank}.npy"), ye)
    # timing reduction
    got = dist.max_over_ranks(10.0 + rank)
    np.save(os.path.join(outdir, f"max_{rank}.npy"), np.array([got]))
    dist.barrier()
    tdist.destroy_process_group()


def test_shard_partitions_exactly():
    for n in (0, 1, 7, 15, 7168):
        for size in (1, 2, 3, 8):
            spans = [dist.shard(n, r, size) for r in range(size)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [h - l for l, h in spans]
            assert max(sizes) - min(sizes) <= 1


def test_two_gloo_ranks_match_single_process(tmp_path):
    size = 2
    mp.spawn(_worker, args=(size, _free_port(), str(tmp_path)), nprocs=size, join=True)
    import oracle
    orc = oracle.get()
    x = inputs.instancenorm_large("cpu", shape=(3, 5, 16, 16), seed=77).reshape(15, 256).numpy()
    ref, _, _ = orc.instancenorm(x)
    got = np.concatenate([np.load(tmp_path / f"in_{r}.npy") for r in range(size)])
    assert np.array_equal(got, ref)
    xe, m = inputs.epilogue("cpu", shape=(5, 4, 2, 3, 4), seed=78)
    refe, _, _ = orc.epilogue(xe.numpy(), m.numpy())
    gote = np.concatenate([np.load(tmp_path / f"epi_{r}.npy") for r in range(size)])
    assert np.array_equal(gote, refe)
    assert all(float(np.load(tmp_path / f"max_{r}.npy")[0]) == 11.0 for r in range(size))


def test_max_over_ranks_single_process():
    assert dist.max_over_ranks(3.5) == 3.5
    assert dist.world_from_env().size >= 1


def _chan_merge(a, b):
    """Pairwise (Chan) merge of (n, mean, M2) rows -- test-side arithmetic."""
    n = a[0] + b[0]
    if b[0] == 0:
        return a
    if a[0] == 0:
        return b
    d = b[1] - a[1]
    return (n, a[1] + d * b[0] / n, a[2] + b[2] + d * d * a[0] * b[0] / n)


def _syncbn_worker(rank, size, port, outdir, splits):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=size)
    import oracle
    from normalization_reduction_gb300 import syncbn
    orc = oracle.get()
    x, _, _, _, _ = inputs.batchnorm("cpu", shape=(sum(splits), 4, 5, 10), seed=91)
    lo = sum(splits[:rank])
    shard = x[lo:lo + splits[rank]].numpy()
    C, S = 4, 50
    local = torch.zeros((C, syncbn.STAT_WIDTH), dtype=torch.float32)
    if splits[rank] * S >= 2:
        _, _, _, mean, var = orc.batchnorm_train(shard)
        cnt = splits[rank] * S
        local[:, 0] = cnt
        local[:, 1] = torch.from_numpy(mean).float()
        local[:, 2] = torch.from_numpy(var * cnt).float()
    gathered = syncbn.gather_rank_stats(local)
    np.save(os.path.join(outdir, f"gathered_{rank}.npy"), gathered.numpy())
    np.save(os.path.join(outdir, f"local_{rank}.npy"), local.numpy())
    tdist.destroy_process_group()


def test_syncbn_exchange_gloo(tmp_path):
    """Three gloo ranks (one with an empty shard) gather per-channel (n, mean, M2)
    in rank order; merged in that order they give the whole batch's statistics."""
    splits = [3, 0, 5]
    size = len(splits)
    mp.spawn(_syncbn_worker, args=(size, _free_port(), str(tmp_path), splits), nprocs=size,
             join=True)
    g = [np.load(tmp_path / f"gathered_{r}.npy") for r in range(size)]
    loc = [np.load(tmp_path / f"local_{r}.npy") for r in range(size)]
    for r in range(size):
        assert g[r].shape == (size, 4, 4)
        assert np.array_equal(g[r], g[0])              # every rank sees the same array
        assert np.array_equal(g[0][r], loc[r])         # row r is rank r's statistics
    import oracle
    orc = oracle.get()
    x, _, _, _, _ = inputs.batchnorm("cpu", shape=(sum(splits), 4, 5, 10), seed=91)
    _, _, _, mean, var = orc.batchnorm_train(x.numpy())
    for c in range(4):
        acc = (0.0, 0.0, 0.0)
        for r in range(size):
            row = g[0][r, c].astype(np.float64)
            acc = _chan_merge(acc, (row[0], row[1], row[2]))
        assert acc[0] == sum(splits) * 50
        assert abs(acc[1] - mean[c]) <= 1e-6 * max(1.0, abs(mean[c]))
        assert abs(acc[2] / acc[0] - var[c]) <= 1e-5 * var[c]


def _dead_peer_worker(rank, size, port, outdir):
    import datetime
    import time
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=size,
                             timeout=datetime.timedelta(seconds=5))
    from normalization_reduction_gb300 import syncbn
    if rank == 1:
        return                      # leaves without joining the gather
    t0 = time.monotonic()
    try:
        syncbn.gather_rank_stats(torch.zeros((4, syncbn.STAT_WIDTH)))
        outcome = "returned"
    except Exception as e:          # the gather must fail, not hang
        outcome = "raised " + type(e).__name__
    with open(os.path.join(outdir, "outcome.txt"), "w") as f:
        f.write(f"{outcome} {time.monotonic() - t0:.1f}")


def test_gather_fails_when_a_rank_leaves(tmp_path):
    """A rank that leaves before the statistics exchange: the other rank's
    gather raises within the process-group timeout instead of hanging."""
    mp.spawn(_dead_peer_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    outcome, secs = open(tmp_path / "outcome.txt").read().rsplit(" ", 1)
    assert outcome.startswith("raised"), outcome
    assert float(secs) < 60
