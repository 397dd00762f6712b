"""Multi-rank host logic on CPU (gloo, world size 2): the slowest-rank reduction the
benchmark uses, and request sharding across ranks (no data-path collective)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from speculative_decoding_draft_rmsnorm_gb300 import workloads as W
from speculative_decoding_draft_rmsnorm_gb300.sharding import shard_requests


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import torch
    import torch.distributed as dist
    from speculative_decoding_draft_rmsnorm_gb300.sharding import max_over_ranks, shard_requests
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = max_over_ranks(10.0 + 5.0 * rank)
        lens = W.context_lengths(W.CONFIGS["ragged"])
        mine = shard_requests(lens, np.full(len(lens), 16), world)[rank]
        t = torch.tensor([float(lens[mine].sum() + 16 * len(mine))], dtype=torch.float64)
        dist.all_reduce(t)
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(f"{got} {t.item()} {','.join(map(str, mine))}\n")
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_sharded_totals(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    lens = W.context_lengths(W.CONFIGS["ragged"])
    rows = [open(tmp_path / f"r{r}.txt").read().split() for r in range(2)]
    for got, total, _ in rows:
        assert float(got) == 15.0                      # every rank sees the slowest time
        assert float(total) == lens.sum() + 16 * len(lens)  # shards cover the batch once
    owned = sorted(int(x) for _, _, idx in rows for x in idx.split(","))
    assert owned == list(range(len(lens)))


@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_shard_balance(world):
    lens = W.context_lengths(W.CONFIGS["ragged"])
    blocks = np.full(len(lens), 16)
    shards = shard_requests(lens, blocks, world)
    assert sorted(np.concatenate(shards).tolist()) == list(range(len(lens)))
    load = [int((lens[s] + 16).sum()) for s in shards]
    assert max(load) - (sum(load) / world) <= int((lens + 16).max())
