"""The multi-rank logic of bench.py on CPU: two gloo ranks (as torchrun would start them) agree on the
maximum of their timings, pass the barrier, and only rank 0 runs and prints the reference arm and the
--extras line."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        out[rank] = bench.max_over_ranks(1.5 + rank, world)
        if rank != 0:  # the reference arm and --extras: every rank but 0 exits at once, without work or output
            out[world + rank] = float(bench.run_reference(type("A", (), {"steps": 1, "warmup": 0})()))
            out[2 * world + rank] = float(bench.run_extras(type("A", (), {"steps": 1, "warmup": 3, "rows": ""})()))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_gate_the_reference_arm():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    assert out[0] == pytest.approx(2.5) and out[1] == pytest.approx(2.5)
    assert out[world + 1] == 0.0
    assert out[2 * world + 1] == 0.0
