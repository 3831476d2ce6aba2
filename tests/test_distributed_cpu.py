"""The multi-rank host logic of bench.py on CPU (gloo, world size 2). The
path partitions into independent (batch, KV head) problems with no exchange
step, and each GPU machine has one GPU, so N GPUs run N independent replicas;
the only cross-rank operations are the timing barrier and the max-over-ranks
reduction of the step time. Both are checked here without a GPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    t = bench.max_over_ranks(10.0 * (rank + 1), w)
    bench.barrier(w)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(repr(t))
    dist.destroy_process_group()


def test_barrier_and_max_over_ranks_with_gloo(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    vals = [float(open(tmp_path / f"rank{r}.txt").read()) for r in range(world)]
    assert vals == [20.0, 20.0]


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    assert bench.dist_setup() == (1, 0, 0)
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
