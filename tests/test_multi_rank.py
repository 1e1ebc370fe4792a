"""Multi-rank host logic of bench.py, run as world-size-2 gloo ranks on the CPU.

The path shards by sequence (independent auctions), so N GPUs run N replicas
with no collective on the data path; the only exchange is the max over ranks of
the step time, which these tests exercise with two CPU processes.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as tmp

import bench
from synth import workloads as W


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, vals, out_dir):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        got = bench.max_over_ranks(vals[rank], world)
        ref = bench.run_reference(_Args(), W.get_config("tiny"), rank, world)
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(" ".join(repr(x) for x in got) + "\n")
            f.write("none\n" if ref is None else "line\n")
        dist.barrier()
    finally:
        dist.destroy_process_group()


class _Args:
    steps = 1
    warmup = 0
    decode_steps = 1


def test_two_ranks_agree_on_the_slowest_step(tmp_path):
    vals = [[12.5, 40.0], [17.25, 31.0]]
    tmp.start_processes(_rank_main, args=(2, _free_port(), vals, str(tmp_path)), nprocs=2,
                        join=True, start_method="spawn")
    for r in range(2):
        lines = open(tmp_path / f"r{r}.txt").read().split("\n")
        assert [float(x) for x in lines[0].split()] == [17.25, 40.0]
        # the reference arm runs on rank 0 only; other ranks exit without work
        assert lines[1] == ("line" if r == 0 else "none")


def test_single_rank_max_is_identity():
    assert bench.max_over_ranks([3.0, 4.5], 1) == [3.0, 4.5]


def test_job_throughput_counts_every_replica():
    # two replicas of 16384 tokens whose slowest step takes 50 ms
    assert bench.job_throughput(16384, 2, 50.0) == pytest.approx(2 * 16384 / 0.05)


def test_replicas_draw_distinct_workloads():
    cfg = W.get_config("tiny")
    a = W.make_workload(bench.replica_config(cfg, 0))
    b = W.make_workload(bench.replica_config(cfg, 1))
    assert bench.replica_config(cfg, 0).seed == cfg.seed
    assert not np.array_equal(a.seqs[0].K, b.seqs[0].K)


def test_parallel_workload_builder_is_the_serial_one():
    cfg = W.small_config(B=2, L=2, H=2, n=700, n_min=500)
    a, b = W.make_workload(cfg), W.make_workload_parallel(cfg, 2)
    for x, y in zip(a.seqs, b.seqs):
        assert np.array_equal(x.K, y.K) and np.array_equal(x.V, y.V) and np.array_equal(x.Qp, y.Qp)
        assert x.needles == y.needles and np.array_equal(x.slot_bounds, y.slot_bounds)
