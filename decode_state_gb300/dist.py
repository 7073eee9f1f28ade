"""Multi-process plumbing: one process per GPU, launched by torch.distributed.run.

The SDM decode shards without any exchange: streams own private bank rows, so a job of S streams
splits into contiguous stream ranges, each rank holding its streams' bank rows and inputs and
running the same kernel on them (stream_shard). The only collectives are the host-side barrier
and the max-over-ranks of the timed region.
"""

from __future__ import annotations

import dataclasses
import os

import torch
import torch.distributed as dist


@dataclasses.dataclass(frozen=True)
class Rank:
    rank: int
    world: int
    local_rank: int

    @property
    def is_root(self) -> bool:
        return self.rank == 0


def init_from_env(backend: str | None = None) -> Rank:
    """Join the process group described by RANK / WORLD_SIZE / MASTER_ADDR / MASTER_PORT (if any)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    if world > 1 and not dist.is_initialized():
        if backend is None:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return Rank(rank, world, local)


def barrier(r: Rank, device=None):
    if r.world > 1:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(r: Rank, value: float, device=None) -> float:
    if r.world == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(r: Rank, value: float, device=None) -> float:
    if r.world == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def shard_seed(base_seed: int, r: Rank) -> int:
    """A seed of this rank's own, for workloads that are not split (each rank draws its own)."""
    return base_seed + 1000003 * r.rank


def shard_range(n: int, r: Rank) -> tuple[int, int]:
    """Contiguous split of n units over the ranks (sizes differ by at most one)."""
    base, extra = divmod(n, r.world)
    lo = r.rank * base + min(r.rank, extra)
    return lo, lo + base + (1 if r.rank < extra else 0)


def stream_shard(n_streams: int, r: Rank, block: int) -> tuple[int, int]:
    """This rank's streams [lo, hi) of an n_streams job split on `block`-stream boundaries: the
    blocks are split as evenly as shard_range splits units (the last block may be shorter)."""
    nb = (n_streams + block - 1) // block
    b0, b1 = shard_range(nb, r)
    return min(b0 * block, n_streams), min(b1 * block, n_streams)


def shutdown(r: Rank):
    if r.world > 1 and dist.is_initialized():
        dist.destroy_process_group()
