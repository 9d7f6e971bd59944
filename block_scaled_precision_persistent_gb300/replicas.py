"""Host-side multi-process plumbing: one process per GPU, independent replicas.

The GEMM shards with no exchange: output tiles are independent, so a job of
several GEMMs (or one GEMM split by output columns) runs as unchanged
single-GPU calls, one per rank. What crosses ranks is only the timing
(barrier, max over ranks) and, for a column-split GEMM, an optional gather of
the BF16 column blocks. Nothing here touches the data path of a kernel.
"""
from __future__ import annotations

import os

import torch


class Ranks:
    """Rank / world from the launcher's environment (RANK, WORLD_SIZE,
    LOCAL_RANK, MASTER_ADDR/PORT). backend: "nccl" on GPUs, "gloo" on CPU.
    With WORLD_SIZE 1 no process group is created and every collective is
    the identity."""

    def __init__(self, backend: str = "nccl", expected_world: int | None = None):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", str(self.rank)))
        if expected_world is not None and self.world != expected_world:
            raise SystemExit(f"expected {expected_world} ranks but WORLD_SIZE={self.world}")
        self.backend = backend
        self.pg = False
        if self.world > 1:
            import torch.distributed as dist
            if backend == "nccl":
                dist.init_process_group("nccl", device_id=torch.device("cuda", self.local))
            else:
                dist.init_process_group(backend)
            self.pg = True

    def _device(self):
        return torch.device("cuda", self.local) if self.backend == "nccl" else torch.device("cpu")

    def barrier(self) -> None:
        if self.pg:
            import torch.distributed as dist
            dist.barrier()

    def max(self, x: float) -> float:
        """The largest x over all ranks (a job is as slow as its slowest rank)."""
        if not self.pg:
            return x
        import torch.distributed as dist
        t = torch.tensor([x], dtype=torch.float64, device=self._device())
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if not self.pg:
            return x
        import torch.distributed as dist
        t = torch.tensor([x], dtype=torch.float64, device=self._device())
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        return float(t.item())

    def gather_columns(self, block: torch.Tensor, n_total: int) -> torch.Tensor:
        """All-gather each rank's [M, n_r] column block (shard_range order)
        into the full [M, n_total] matrix on every rank."""
        if not self.pg:
            return block
        import torch.distributed as dist
        m = block.shape[0]
        widths = [shard_range(n_total, self.world, r)[1] - shard_range(n_total, self.world, r)[0]
                  for r in range(self.world)]
        wmax = max(widths)
        pad = torch.zeros((m, wmax), dtype=block.dtype, device=block.device)
        pad[:, :block.shape[1]] = block
        parts = [torch.empty_like(pad) for _ in range(self.world)]
        dist.all_gather(parts, pad)
        return torch.cat([p[:, :w] for p, w in zip(parts, widths)], dim=1)

    def close(self) -> None:
        if self.pg:
            import torch.distributed as dist
            dist.destroy_process_group()
            self.pg = False


def shard_range(n: int, world: int, rank: int, align: int = 8) -> tuple[int, int]:
    """Contiguous [n0, n1) block of n output columns for `rank` of `world`,
    block edges on multiples of `align` (the GEMM requires N % 8 == 0 per
    call, and a B shard then starts on a 16-byte boundary for any K the GEMM
    accepts). Blocks differ in size by at most `align`; trailing ranks may
    get an empty block when n is small."""
    if n < 0 or world < 1 or not 0 <= rank < world or align < 1:
        raise ValueError("bad shard arguments")
    units = -(-n // align)
    u0 = units * rank // world
    u1 = units * (rank + 1) // world
    return min(n, u0 * align), min(n, u1 * align)
