"""Replicas across GPUs of one node: one process per GPU, each running the whole
layer on its own batch (the (sequence, head) units are independent, so the work
shards by batch with no exchange on the data path).  Only the timing needs the
ranks together: a barrier on both sides of the timed region and the maximum of
the per-rank times.

Launch: ``python -m torch.distributed.run --nproc-per-node N ...`` (RANK,
LOCAL_RANK, WORLD_SIZE and MASTER_ADDR/PORT from the environment), or one plain
process (world size 1, no process group).
"""
from __future__ import annotations

import os
from dataclasses import dataclass
from typing import Optional


@dataclass
class Replicas:
    world: int = 1
    rank: int = 0
    local_rank: int = 0
    backend: Optional[str] = None   # None until init(): no process group

    @classmethod
    def from_env(cls) -> "Replicas":
        return cls(int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
                   int(os.environ.get("LOCAL_RANK", "0")))

    @property
    def is_root(self) -> bool:
        return self.rank == 0

    def seed(self, base: int = 0) -> int:
        """Seed of this rank's synthetic batch (each replica draws its own)."""
        return base + self.rank

    def init(self, backend: str, device=None) -> None:
        """Join the process group (nccl with a CUDA device, gloo on the CPU) when
        there is more than one rank."""
        if self.world <= 1:
            return
        import torch.distributed as dist
        if device is not None and backend == "nccl":
            dist.init_process_group(backend, device_id=device)
        else:
            dist.init_process_group(backend)
        self.backend = backend

    def barrier(self) -> None:
        if self.backend:
            import torch.distributed as dist
            dist.barrier()

    def max_over_ranks(self, value: float, device=None) -> float:
        """The largest of the ranks' values (the job's time is its slowest replica's)."""
        if not self.backend:
            return float(value)
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(value)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def total_units(self, per_rank: int) -> int:
        """Units processed by the whole job (every replica does the same amount)."""
        return per_rank * self.world

    def shutdown(self) -> None:
        if self.backend:
            import torch.distributed as dist
            dist.destroy_process_group()
            self.backend = None
