"""The N > 1 path of bench.py on CPU: two gloo ranks.

Attention shards into independent (sequence, head) problems, so several GPUs
run independent replicas and the only cross-rank step is the timing
aggregation (a barrier and the max over ranks of the elapsed time).  These
tests exercise exactly that code with the gloo backend, no GPU needed.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      FA_BENCH_BACKEND="gloo")
    import sys
    sys.path.insert(0, ROOT)
    import bench
    r, w = bench.dist_init(world)
    assert (r, w) == (rank, world)
    bench.barrier(w)
    ms = [12.5, 20.0][rank]                      # rank 1 is the slow one
    slowest = bench.max_over_ranks(ms, w)
    value = bench.aggregate_tflops(1e12, 10, w, slowest)
    out[rank] = (slowest, value)
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_by_the_slowest_rank():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0] == out[1]
    slowest, value = out[0]
    assert slowest == 20.0
    # 2 ranks x 10 steps x 1 TFLOP in 20 ms
    assert value == pytest.approx(2 * 10 * 1.0 / 0.020)


def test_single_rank_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.aggregate_tflops(2e12, 5, 1, 10.0) == pytest.approx(1000.0)
