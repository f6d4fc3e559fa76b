"""CPU, world size 2 over gloo: the bench's multi-rank host logic (barrier, max over ranks of the
timed region, weak-scaling aggregate).  The path shards by independent layers, one per rank, with
no data-path collective; only the timing uses torch.distributed."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, lr = bench.dist_env()
    assert (w, r, lr) == (world, rank, rank)
    d = bench.dist_init(w, torch.device("cpu"))
    bench.barrier(d, torch.device("cpu"))
    ms = 10.0 + 5.0 * rank  # rank 1 is the slowest
    ms_max = bench.max_over_ranks(d, ms, torch.device("cpu"))
    out[rank] = ms_max
    d.destroy_process_group()


def test_max_over_ranks_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 15.0


def test_weak_scaling_aggregate():
    # two ranks, each 1.9e12 flops per step, 10 steps, slowest rank 20 ms -> 1900 TFLOP/s
    assert bench.aggregate_tflops(2, 1.9e12, 10, 20.0) == pytest.approx(1900.0)
    assert bench.aggregate_tflops(1, 1.9e12, 10, 20.0) == pytest.approx(950.0)


def test_single_rank_needs_no_process_group():
    assert bench.dist_init(1, torch.device("cpu")) is None
    assert bench.max_over_ranks(None, 3.5, torch.device("cpu")) == 3.5


def test_visible_pairs_closed_form():
    import itertools

    for N, W in itertools.product((1, 5, 17, 128), (1, 2, 7, 128, 500)):
        brute = sum(1 for i in range(N) for j in range(N) if 0 <= i - j < W)
        assert bench.visible_pairs(N, W) == brute


def test_window_pairs_counts_the_mask():
    """The bench's pair count for Lq <= Lk and two-sided windows is the number of visible cells
    (brute-force double loop over the offset window)."""
    import itertools

    for Lq, Lk, W, causal in itertools.product((1, 5, 17), (17, 40), (1, 3, 16, 100),
                                              (True, False)):
        off = Lk - Lq
        brute = sum(1 for i in range(Lq) for j in range(Lk)
                    if (0 <= i + off - j < W if causal else abs(i + off - j) < W))
        assert bench.window_pairs(Lq, Lk, W, causal) == brute
    assert bench.window_pairs(300, 300, 64, True) == bench.visible_pairs(300, 64)
