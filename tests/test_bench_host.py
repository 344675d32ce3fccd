"""Host logic of the multi-rank benchmark (weak scaling, max over ranks),
exercised with two gloo ranks on the CPU."""
from __future__ import annotations

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from speculative_verify_attention_kv_gb300 import workloads as wl
    assert bench.rank_info() == (rank, world, rank)
    bench.barrier(world)
    t = bench.reduce_max(1.0 + rank * 2.5, world)
    spec = wl.SPEC_BY_NAME["tiny"]
    seeds = [bench.rank_seed(spec, r) for r in range(world)]
    W = wl.Workload(spec, bench.rank_seed(spec, rank))
    out[rank] = (t, seeds, int(W.q_bits()[0, 0, 0]))
    dist.destroy_process_group()


def test_two_rank_max_reduction_and_independent_batches():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == pytest.approx(3.5)       # max over ranks
    assert res[0][1] == res[1][1] and len(set(res[0][1])) == 2  # distinct seeds per rank
    assert res[0][2] != res[1][2]                                # different data per rank


def test_launch_count_matches_the_kernels_a_step_runs():
    sys.path.insert(0, ROOT)
    import bench
    from speculative_verify_attention_kv_gb300 import workloads as wl
    W = wl.make("batch16_32k")
    n = bench.dw_launches_per_step(W, 0)
    assert n == 4
