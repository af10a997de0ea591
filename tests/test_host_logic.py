"""Host-side logic of the benchmark and the input recipe (no GPU)."""
import os
import socket

import numpy as np
import pytest
import torch

import bench
from attention_fa2_forward_gb300.inputs import WORKLOADS, make_qkv, workload_inputs


def _brute_pairs(S, causal, window):
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    vis = np.ones((S, S), dtype=bool)
    if causal:
        vis &= j <= i
    if window > 0:
        vis &= (i - j) < window
        if not causal:
            vis &= (j - i) < window
    return int(vis.sum()), vis.sum(axis=1)


@pytest.mark.parametrize("S,causal,window", [(1, False, -1), (7, True, -1), (9, True, 1),
                                             (33, True, 5), (40, True, 40), (41, True, 60),
                                             (17, False, -1), (17, False, 1), (33, False, 5),
                                             (20, False, 20), (20, False, 19), (7, False, 100)])
def test_visible_pair_count_matches_brute_force(S, causal, window):
    total, per_row = _brute_pairs(S, causal, window)
    assert bench.visible_pairs(S, causal, window) == total
    for i in range(S):
        assert bench.visible_keys_of_row(i, S, causal, window) == per_row[i]


def test_workload_flops_match_the_published_shapes():
    # 4 * B * H * D * pairs, pairs counted exactly.
    w = WORKLOADS["gqa_s4096_d128"]
    assert bench.workload_flops(w) == 4 * 2 * 32 * 128 * (4096 * 4097 // 2)
    w = WORKLOADS["swa_s16384_w4096"]
    assert bench.workload_flops(w) == 4 * 32 * 128 * (4096 * 4097 // 2 + (16384 - 4096) * 4096)


def test_oracle_sample_rows_spread_and_bounded():
    w = WORKLOADS["mqa_s32768_stress"]
    rows = bench.oracle_sample_rows(w, 5e9)
    assert rows == sorted(set(rows)) and 0 <= rows[0] and rows[-1] < w.S
    assert len(rows) >= 2
    assert bench.sampled_flops(w, rows) <= 2 * 5e9
    assert bench.oracle_sample_rows(WORKLOADS["tiny_f32"], 1e12) == list(range(128))


def test_inputs_are_seeded_and_rounded():
    a = make_qkv(1, 8, 2, 1, 64, torch.bfloat16, seed=3)
    b = make_qkv(1, 8, 2, 1, 64, torch.bfloat16, seed=3)
    c = make_qkv(1, 8, 2, 1, 64, torch.bfloat16, seed=4)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert not torch.equal(a[0], c[0])
    q, k, v = a
    assert q.shape == (1, 8, 2, 64) and k.shape == (1, 8, 1, 64) and v.dtype == torch.bfloat16
    # bf16 values are the round-to-nearest-even images of the fp32 draws.
    g = torch.Generator().manual_seed(3)
    q32 = torch.randn((1, 8, 2, 64), generator=g)
    assert torch.equal(q, q32.to(torch.bfloat16))


def test_stress_workload_distribution():
    w = WORKLOADS["mqa_s32768_stress"]
    q, k, v = workload_inputs(w, S=512)
    assert 2.5 < q.float().std().item() < 3.5 and 2.5 < k.float().std().item() < 3.5
    assert v.float().abs().max().item() <= 1.0


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist = bench.init_dist(world, "gloo")
    value = bench.max_over_ranks(float(10 * (rank + 1)), dist)
    bench.barrier(dist)
    out[rank] = value
    dist.destroy_process_group()


def test_timing_is_max_reduced_over_ranks():
    """bench.py's multi-rank helpers: every rank sees the slowest rank's time."""
    import torch.multiprocessing as mp
    world = 2
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    assert dict(out) == {0: 20.0, 1: 20.0}
