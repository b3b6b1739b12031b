"""Multi-GPU replicas, host side: two gloo ranks on CPU exercise the
benchmark's aggregation (slowest rank's time, whole-job throughput) and the
per-rank input seeding, without a GPU."""
import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from draft_head_gb300 import synth


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 100.0 + 50.0 * rank  # rank 1 is the slowest replica
    m = bench.max_over_ranks(ms, dist, "cpu")
    v = bench.replica_throughput(15 * 10, world, m)
    seed = synth.case_seed("tiny_f32", 0) + 7919 * rank
    H = synth.make_case(synth.CONFIGS["tiny_f32"], seed)["H"]
    out[rank] = (m, v, float(H.sum()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replica_aggregation():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 150.0
    assert abs(res[0][1] - 2 * 150 / 0.150) < 1e-6
    assert res[0][2] != res[1][2]  # each replica drafts its own inputs
