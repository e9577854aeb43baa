"""Multi-process helpers (one process per GPU).

InstanceNorm and the fused epilogue are independent per slice / per sample,
so running them on several GPUs needs no collective on the data path: each
rank takes a contiguous shard of the units (or, in the benchmark, its own
replica of the workload), and the only communication is a barrier and a
max-reduction of the measured times. These helpers work with any
``torch.distributed`` backend (NCCL across GPUs, gloo on the CPU in tests).
"""
from __future__ import annotations

import os
from dataclasses import dataclass

import torch
import torch.distributed as tdist


@dataclass(frozen=True)
class World:
    rank: int
    size: int
    local_rank: int


def world_from_env() -> World:
    """RANK / WORLD_SIZE / LOCAL_RANK as set by torchrun (defaults: one process)."""
    return World(int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
                 int(os.environ.get("LOCAL_RANK", "0")))


def shard(n_units: int, rank: int, size: int) -> tuple[int, int]:
    """Contiguous, balanced share [lo, hi) of n_units for `rank` of `size`:
    the first n_units % size ranks get one unit more."""
    if size < 1 or not 0 <= rank < size or n_units < 0:
        raise ValueError("bad shard request")
    base, extra = divmod(n_units, size)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def max_over_ranks(value: float, device=None) -> float:
    """The maximum of `value` over all ranks (the value itself when
    torch.distributed is not initialised)."""
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def barrier() -> None:
    if tdist.is_available() and tdist.is_initialized() and tdist.get_world_size() > 1:
        tdist.barrier()


def free_port() -> int:
    """A TCP port on 127.0.0.1 that was free a moment ago."""
    import socket
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch_plan(gpus: int, environ, argv, script: str, python: str, port: int | None = None):
    """How a benchmark asked to run on ``gpus`` GPUs (one process each) starts.

    * not under a launcher (no WORLD_SIZE) and gpus == 1: run here, one rank;
    * not under a launcher and gpus > 1: re-launch the same command line under
      ``torch.distributed.run`` with one process per GPU on 127.0.0.1;
    * under a launcher: run here when WORLD_SIZE equals gpus, else an error.

    Returns a dict with "action" in {"run", "relaunch", "error"} and, for
    "run", the world size; for "relaunch", the command; for "error", why.
    """
    if gpus < 1:
        return {"action": "error", "why": f"--gpus must be >= 1 (got {gpus})"}
    ws = environ.get("WORLD_SIZE")
    if ws is None:
        if gpus == 1:
            return {"action": "run", "world_size": 1}
        cmd = [python, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={gpus}",
               "--master-addr", "127.0.0.1", "--master-port", str(port or free_port()), script,
               *argv]
        return {"action": "relaunch", "cmd": cmd, "world_size": gpus}
    if int(ws) != gpus:
        return {"action": "error",
                "why": f"launched with WORLD_SIZE={ws} processes but --gpus {gpus}"}
    return {"action": "run", "world_size": gpus}
