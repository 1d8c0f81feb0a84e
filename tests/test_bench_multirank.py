"""World-size-2 gloo test of the bench's multi-rank logic on CPU: independent replicas (distinct
seeded batches, no data-path collective), timings reduced by max over ranks, and the whole-job
value counting every rank's work."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from attention_backward_fabwd_gb300 import inputs

    mine = [1.0 + rank, 5.0 - rank, 2.0 * rank]
    got = bench.max_over_ranks(mine, world)
    w = bench.replica_workload(inputs.WORKLOADS["mha_s128_d64"], rank)
    pb = inputs.make_problem(w)
    out[rank] = (got, w.seed, float(pb.q.float().sum()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_replicas():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    (g0, s0, q0), (g1, s1, q1) = res[0], res[1]
    assert g0 == g1 == [2.0, 5.0, 2.0]
    assert s0 != s1 and q0 != q1


def test_job_value_counts_all_ranks():
    import bench

    assert bench.job_tflops(1e12, 2, 1000.0) == pytest.approx(2.0)
    assert bench.job_tflops(3e12, 1, 1500.0) == pytest.approx(2.0)
