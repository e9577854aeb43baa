"""Synchronised (multi-process) training BatchNorm over the library's C ABI.

Each process holds a shard of the batch (along N) on its own GPU. The only
communication is one all-gather of the per-channel statistics (count, mean,
M2) -- C x 16 bytes per rank -- between the two library calls:

    fnorm_batchnorm_local_stats  (GPU)  ->  all_gather over the process group
    ->  fnorm_batchnorm_apply_stats (GPU: rank-order merge, normalise, running
        statistics)

so every rank normalises its shard with the statistics of the whole batch.
"""
from __future__ import annotations

import torch
import torch.distributed as tdist

from . import fnorm_batchnorm_apply_stats, fnorm_batchnorm_local_stats
from . import fnorm_batchnorm_workspace_size

STAT_WIDTH = 4   # (count, mean, M2, unused) per channel


def gather_rank_stats(local: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather the [C][4] statistics of every rank into [R][C][4], rank order."""
    if not (tdist.is_available() and tdist.is_initialized()):
        return local.unsqueeze(0).contiguous()
    world = tdist.get_world_size(group)
    if world == 1:
        return local.unsqueeze(0).contiguous()
    parts = [torch.empty_like(local) for _ in range(world)]
    tdist.all_gather(parts, local.contiguous(), group=group)
    return torch.stack(parts).contiguous()


def sync_batch_norm_train(x, gamma=None, beta=None, running_mean=None, running_var=None,
                          momentum: float = 0.1, eps: float = 1e-5, scale: float = 1.0,
                          group=None, workspace=None, out=None, stream=None):
    """Training BatchNorm of this rank's shard x [N, C, *spatial] (fp32, CUDA)
    with statistics over all ranks' shards; returns y (the shard's output)."""
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor")
    N, C = x.shape[0], x.shape[1]
    S = 1
    for d in x.shape[2:]:
        S *= d
    nbytes = fnorm_batchnorm_workspace_size(N, C, S)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=x.device)
    local = torch.empty((C, STAT_WIDTH), dtype=torch.float32, device=x.device)
    fnorm_batchnorm_local_stats(x, local, N, C, S, workspace, workspace.numel(), stream)
    stats_all = gather_rank_stats(local, group)
    y = out if out is not None else torch.empty_like(x)
    fnorm_batchnorm_apply_stats(x, y, stats_all, stats_all.shape[0], gamma, beta, scale,
                                running_mean, running_var, momentum, eps, None, None, N, C, S,
                                stream)
    return y
