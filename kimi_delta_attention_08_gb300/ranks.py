"""Host-side rank logic for multi-GPU runs of the forward.

(sequence, head) units are independent, so N GPUs run N independent batches
(weak scaling): rank r draws its own inputs (seed offset r) and nothing on the
data path is exchanged.  The only cross-rank traffic is timing: a barrier on
both sides of the timed region and the maximum step time over ranks.
These helpers take the process group as an argument so the same code runs
over NCCL on GPUs and over gloo on CPU.
"""
from __future__ import annotations

import os
import socket
import subprocess
import sys


def world_info():
    """(rank, world_size, local_rank) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(base_seed: int, rank: int) -> int:
    """Input seed of rank `rank`: every rank processes a distinct batch."""
    return base_seed + 1000 * rank


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The largest value of `x` over all ranks (the job's step time)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tokens_per_s(tokens_per_rank: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: the tokens every rank processed over the slowest rank's time."""
    return tokens_per_rank * world / (max_ms * 1e-3)


def free_port() -> int:
    """An unused TCP port on 127.0.0.1 for the rendezvous."""
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def spawn_world(nproc: int, argv, port: int | None = None) -> int:
    """Run `argv` (a script and its arguments) as `nproc` processes on this node,
    one per GPU, through torch.distributed.run with the rendezvous on 127.0.0.1;
    each process finds RANK, LOCAL_RANK and WORLD_SIZE in its environment.
    Returns the launcher's exit code (non-zero if any rank failed)."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={int(nproc)}", "--master-addr=127.0.0.1",
           f"--master-port={port or free_port()}"] + [str(a) for a in argv]
    return subprocess.run(cmd).returncode
