"""bench.py's reductions over ranks (the N > 1 launch: one process per GPU,
max of the timed region over ranks, tokens summed over ranks), checked with
two and three gloo ranks on CPU."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, path):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        mx = bench.max_over_ranks(dist, 10.0 + rank)          # e.g. elapsed ms per rank
        sm = bench.sum_over_ranks(dist, 64.0 * (rank + 1))    # tokens per rank
        bench.barrier(dist)
        if rank == 0:
            torch.save({"max": mx, "sum": sm}, path)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_rank_reductions(tmp_path, world):
    path = str(tmp_path / "r.pt")
    mp.start_processes(_rank_main, args=(world, _free_port(), path), nprocs=world, join=True,
                       start_method="spawn")
    r = torch.load(path)
    assert r["max"] == 10.0 + world - 1
    assert r["sum"] == 64.0 * world * (world + 1) / 2


def test_single_process_reductions_are_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 3.5) == 3.5 and bench.sum_over_ranks(None, 7.0) == 7.0
