"""bench.py's multi-rank host logic on CPU: two gloo ranks, max-over-ranks time and
whole-job throughput (no GPU; the data path itself has no collective)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [3.0, 5.5][rank]
        worst = bench.max_over_ranks(mine, dist, torch.device("cpu"))
        out[rank] = worst
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_value():
    sys.path.insert(0, ROOT)
    import bench
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, start_method="spawn", join=True)
    assert out[0] == 5.5 and out[1] == 5.5
    # two ranks of 1e12 FLOPs each, slowest rank 5.5 ms -> 2e12 / 5.5e-3 s
    assert bench.whole_job_tflops(1e12, 2, 5.5) == pytest.approx(2e12 / 5.5e-3 / 1e12)
    assert bench.max_over_ranks(4.0, None, torch.device("cpu")) == 4.0


def test_flop_and_byte_counts():
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    from workloads import WORKLOADS
    w = WORKLOADS[5]
    assert bench.nominal_flops(w) == 4.0 * 4 * 16 * 8192 * 8192 * 64 / 2
    assert bench.useful_flops(w, np.full(4, 8192)) == 4.0 * 64 * 4 * 16 * 8192 * 8193 / 2
    w3 = WORKLOADS[3].with_(B=1, h=1, m=3, n=3)
    assert bench.allowed_pairs(w3, [3]) == 6                       # 1 + 2 + 3
    w2 = WORKLOADS[2].with_(B=2, h=1, m=4, n=4)
    assert bench.allowed_pairs(w2, [1, 3]) == 4 * 1 + 4 * 3
    rows = np.arange(2 * 4)
    assert bench.row_pairs(w2, [1, 3], rows) == 4 * 1 + 4 * 3
