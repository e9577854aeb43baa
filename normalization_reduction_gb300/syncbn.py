"""Synchronised (multi-process) training BatchNorm over the library's C ABI.

Each process holds a shard of the batch (along N) on its own GPU. The only
communication is one all-gather of the per-channel statistics (count, mean,
M2) -- C x 16 bytes per rank -- between the two library calls:

    fnorm_batchnorm_local_stats  (GPU)  ->  all_gather over the process group
    ->  fnorm_batchnorm_apply_stats (GPU: rank-order merge, normalise, running
        statistics)

so every rank normalises its shard with the statistics of the whole batch
(page Kimi-K2.6__l2_p73, block 1: BatchNorm2d's statistics over (N, H, W),
here over the union of the shards).

Stream ordering. Both library calls run on ``stream`` (torch's current stream
when None). The all-gather is issued on torch's current stream (NCCL orders
itself after that stream; with gloo the statistics go through host memory,
which synchronises it). So the caller's stream first waits for the current
stream (the inputs), the current stream then waits for the statistics kernel
before the gather, and the caller's stream waits for the gather before the
normalisation. Buffers allocated here on the current stream are marked as used
on ``stream`` (``record_stream``) so that the caching allocator does not hand
them out again while the kernels still run. The returned y is complete once
``stream`` reaches this point.
"""
from __future__ import annotations

import torch
import torch.distributed as tdist

from . import fnorm_batchnorm_apply_stats, fnorm_batchnorm_local_stats
from . import fnorm_batchnorm_workspace_size

STAT_WIDTH = 4   # (count, mean, M2, unused) per channel


def _torch_stream(stream, device) -> torch.cuda.Stream:
    if stream is None:
        return torch.cuda.current_stream(device)
    if isinstance(stream, int):
        return torch.cuda.ExternalStream(stream, device=device)
    return stream


def gather_rank_stats(local: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather the [C][4] statistics of every rank into [R][C][4], rank order.

    Runs on torch's current stream. With a backend that cannot gather CUDA
    tensors (gloo), the statistics travel through host memory."""
    if not (tdist.is_available() and tdist.is_initialized()):
        return local.unsqueeze(0).contiguous()
    world = tdist.get_world_size(group)
    if world == 1:
        return local.unsqueeze(0).contiguous()
    if local.is_cuda and tdist.get_backend(group) == "gloo":
        host = local.cpu().contiguous()
        parts = [torch.empty_like(host) for _ in range(world)]
        tdist.all_gather(parts, host, group=group)
        return torch.stack(parts).to(local.device).contiguous()
    parts = [torch.empty_like(local) for _ in range(world)]
    tdist.all_gather(parts, local.contiguous(), group=group)
    return torch.stack(parts).contiguous()


def sync_batch_norm_train(x, gamma=None, beta=None, running_mean=None, running_var=None,
                          momentum: float = 0.1, eps: float = 1e-5, scale: float = 1.0,
                          group=None, workspace=None, out=None, stream=None):
    """Training BatchNorm of this rank's shard x [N, C, *spatial] (fp32, CUDA)
    with statistics over all ranks' shards; returns y (the shard's output).
    ``stream``: a torch.cuda.Stream, a raw cudaStream_t handle, or None for
    torch's current stream."""
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor")
    N, C = x.shape[0], x.shape[1]
    S = 1
    for d in x.shape[2:]:
        S *= d
    cur = torch.cuda.current_stream(x.device)
    work = _torch_stream(stream, x.device)
    separate = work.cuda_stream != cur.cuda_stream
    if separate:
        work.wait_stream(cur)          # inputs written on the current stream
    nbytes = fnorm_batchnorm_workspace_size(N, C, S)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=x.device)
        if separate:
            workspace.record_stream(work)
    local = torch.empty((C, STAT_WIDTH), dtype=torch.float32, device=x.device)
    if separate:
        local.record_stream(work)
    fnorm_batchnorm_local_stats(x, local, N, C, S, workspace, workspace.numel(), work)
    if separate:
        cur.wait_stream(work)          # the gather reads the statistics
    stats_all = gather_rank_stats(local, group)
    y = out if out is not None else torch.empty_like(x)
    if separate:
        work.wait_stream(cur)          # the merge reads the gathered array
        stats_all.record_stream(work)
        if out is None:
            y.record_stream(work)
    fnorm_batchnorm_apply_stats(x, y, stats_all, stats_all.shape[0], gamma, beta, scale,
                                running_mean, running_var, momentum, eps, None, None, N, C, S,
                                work)
    return y
