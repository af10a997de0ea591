"""bench.py's replica path under torchrun (WORLD_SIZE > 1), on CPU with gloo:
every rank reads its place from the environment, the timing reduction takes
the maximum over ranks, and the barriers complete. No GPU is involved (the
GPU arms reduce on NCCL with the same calls)."""
import os
import socket

import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    w, r, local = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    # each rank's "time" differs; every rank must see the maximum
    results[r] = (w, local, bench.max_over_ranks(10.0 + 3.0 * r, dist))
    bench.barrier(dist)
    dist.destroy_process_group()


def test_replica_timing_reduction_over_two_gloo_ranks():
    world = 2
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), results), nprocs=world,
                           join=True, start_method="spawn")
        got = dict(results)
    assert got == {0: (2, 0, 13.0), 1: (2, 1, 13.0)}


def test_single_process_needs_no_process_group():
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(4.5, None) == 4.5
    bench.barrier(None)
