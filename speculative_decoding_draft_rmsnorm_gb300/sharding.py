"""Host-side helpers for running the path on several GPUs.

Requests of a ragged batch are independent (disjoint keys and output rows), so the
path shards by request with no collective on the data path: each rank runs the
library on its own requests. `shard_requests` balances ranks by key count (context +
block rows, the HBM traffic of a request); `max_over_ranks` is the one reduction the
benchmark needs (slowest rank's time).
"""
from __future__ import annotations

import heapq

import numpy as np


def shard_requests(ctx_lens, block_lens, world: int) -> list[np.ndarray]:
    """Longest-processing-time-first assignment of requests to `world` ranks.

    Returns, per rank, the sorted request indices it owns. Every request appears once;
    the heaviest rank exceeds the average load by at most one request's load.
    """
    if world < 1:
        raise ValueError("world must be >= 1")
    load = np.asarray(ctx_lens, np.int64) + np.asarray(block_lens, np.int64)
    heap = [(0, r) for r in range(world)]
    owned: list[list[int]] = [[] for _ in range(world)]
    for i in np.argsort(-load, kind="stable"):
        w, r = heapq.heappop(heap)
        owned[r].append(int(i))
        heapq.heappush(heap, (w + int(load[i]), r))
    return [np.array(sorted(o), dtype=np.int64) for o in owned]


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of a per-rank float over the default process group (identity when alone)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
