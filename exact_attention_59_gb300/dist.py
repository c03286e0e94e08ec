"""Multi-GPU host logic: one process per GPU, no collective on the data path.

Every (b, h) of attention is independent in the forward, the backward and
decode (the attnax Pallas forward launches its grid over (batch, heads,
q blocks) with no communication), so work shards by head with no exchange
step.  The only collectives are for measurement: a barrier around the timed
region and the max of the per-rank times.

* ``shard_heads``: contiguous split of the B*H heads over ranks (strong
  scaling of one batch).
* ``shard_qblocks``: for B*H smaller than the world (the 1 x 2 x 131072
  long-context case), split each head's q blocks, longest causal rows first,
  dealt round-robin so every rank gets a similar number of kv tiles; K/V are
  replicated.
"""

from __future__ import annotations

import os

import torch
import torch.distributed as tdist


def world() -> tuple[int, int]:
    """(rank, world_size) from the torchrun environment (0, 1 without it)."""
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))


def init(backend: str = "nccl") -> tuple[int, int]:
    rank, ws = world()
    if ws > 1 and not tdist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        tdist.init_process_group(backend)
    return rank, ws


def barrier():
    if tdist.is_available() and tdist.is_initialized():
        tdist.barrier()


def max_over_ranks(value: float, device=None) -> float:
    """The largest of the ranks' values (a rank's time), the same on every rank."""
    if not (tdist.is_available() and tdist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def shard_heads(n_heads: int, world_size: int, rank: int) -> range:
    """Contiguous block of heads [lo, hi) of this rank; sizes differ by at most one."""
    base, extra = divmod(n_heads, world_size)
    lo = rank * base + min(rank, extra)
    return range(lo, lo + base + (1 if rank < extra else 0))


def shard_qblocks(nqb: int, world_size: int, rank: int, causal: bool = True) -> list[int]:
    """q blocks of one head for this rank: longest causal rows first, dealt in a
    serpentine order (0,1,..,W-1,W-1,..,0,...) so the kv-tile counts balance."""
    order = list(range(nqb - 1, -1, -1)) if causal else list(range(nqb))
    mine = []
    for i, qb in enumerate(order):
        rnd, pos = divmod(i, world_size)
        owner = pos if rnd % 2 == 0 else world_size - 1 - pos
        if owner == rank:
            mine.append(qb)
    return mine
