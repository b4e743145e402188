"""The multi-rank (replica) path of the benchmark on CPU: two gloo ranks, no GPU.

Requests are independent, so N GPUs serve N disjoint replicas with no collective on the data
path; the process group carries only the barriers and the max-over-ranks of the timings.  This
checks that host logic with world size 2: rank-specific replicas, the max over ranks, and the
whole-job aggregate.
"""
import os
import socket

import numpy as np
import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    r, w = bench.dist_setup(world, backend="gloo", device="cpu")
    wl = bench.rank_workload("decode_b64_fp8_indexshare", r)
    elapsed = 100.0 + 25.0 * r                       # rank 1 is the slow one
    bench.barrier(w)
    mx = bench.max_over_ranks(elapsed, w, device="cpu")
    rate = bench.aggregate_rate(mx, w, wl.layers, 10)
    np.save(os.path.join(out_dir, f"rank{r}.npy"),
            np.array([r, w, mx, rate, wl.seed, wl.num_requests, wl.block_table.sum()], dtype=np.float64))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_serve_disjoint_replicas(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    res = [np.load(tmp_path / f"rank{r}.npy") for r in range(world)]
    for r, x in enumerate(res):
        assert x[0] == r and x[1] == world
        assert x[2] == 125.0                          # both ranks see the slowest rank's time
        assert x[3] == pytest.approx(world * 4 * 10 / 0.125)
        assert x[5] == 64
    assert res[0][4] != res[1][4], "replicas must be drawn from different seeds"
    assert res[0][6] != res[1][6], "replicas must use different page tables"


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
    assert bench.aggregate_rate(500.0, 1, 4, 50) == pytest.approx(400.0)
    wl = bench.rank_workload("decode_b64_fp8_indexshare", 0)
    assert wl.seed == 1003 and wl.layers == 4
