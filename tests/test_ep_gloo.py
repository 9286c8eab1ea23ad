"""Expert-parallel composition on CPU: two gloo ranks each compute the
partial output of their expert range (with the CPU oracle standing in for
the device), sum them with the package's all-reduce, and must reproduce the
whole layer.  No GPU is used."""
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


def _rank_main(rank, world, port, E, result_path):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import gpt_oss_moe_gb300 as moe
    import oracle
    import synth
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        L = synth.make_layer(E=E, T=24, H=64, I=64, top_k=3, seed=71, router_w_std=0.2)
        start, n = moe.ep_expert_range(rank, world, E)
        part = oracle.forward_ep(L, start, n, threads=1)
        total = moe.ep_all_reduce(part.clone())
        if rank == 0:
            _, _, full = oracle.forward(L, threads=1)
            torch.save({"total": total, "full": full}, result_path)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_ep_partials_all_reduce_to_the_layer(tmp_path, world):
    import oracle
    oracle.build()
    path = str(tmp_path / "res.pt")
    mp.start_processes(_rank_main, args=(world, _free_port(), 8, path), nprocs=world,
                       join=True, start_method="spawn")
    res = torch.load(path)
    full, total = res["full"], res["total"]
    assert (total - full).abs().max() <= 1e-6 * full.abs().max()
