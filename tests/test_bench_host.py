"""Host logic of the multi-rank benchmark: the seeded batch partitioned across
ranks by KV bytes, the max-over-ranks timing reduction (two gloo ranks on the
CPU), and the L2 rotation rule."""
from __future__ import annotations

import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from speculative_verify_attention_kv_gb300 import workloads as wl  # noqa: E402


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
    import bench as b
    from speculative_verify_attention_kv_gb300 import workloads as w
    assert b.rank_info() == (rank, world, rank)
    b.barrier(world)
    t = b.reduce_max(1.0 + rank * 2.5, world)
    W = w.make("ragged64")
    seqs = b.rank_sequences(W, world, rank)
    sub = W.subset(seqs)
    out[rank] = (t, list(seqs), int(sub.num_q_tokens), int(sub.q_bits()[0, 0, 0]))
    dist.destroy_process_group()


def test_two_ranks_partition_the_batch_and_reduce_the_time():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == pytest.approx(3.5)       # max over ranks
    W = wl.make("ragged64")
    assert sorted(res[0][1] + res[1][1]) == list(range(W.num_seqs))   # every sequence once
    assert res[0][2] + res[1][2] == W.num_q_tokens
    first = res[0][1][0]                                       # a rank's data is the batch's data
    assert res[0][3] == int(W.q_bits_seq(first)[0, 0, 0])


@pytest.mark.parametrize("name,parts", [("ragged64", 2), ("ragged64", 8), ("batch16_32k", 3),
                                        ("shared_prefix", 2), ("single_32k", 2)])
def test_partition_is_balanced_by_kv_bytes(name, parts):
    W = wl.make(name)
    groups = wl.partition_by_kv_bytes(W, parts)
    assert sorted(sum(groups, [])) == list(range(W.num_seqs))
    cost = W.context_lens.astype(np.int64) + W.block_lens
    loads = [int(cost[g].sum()) for g in groups]
    # greedy largest-first: no group exceeds the mean by more than one sequence
    assert max(loads) <= cost.sum() / parts + cost.max()


def test_subset_keeps_each_sequences_data_and_shares_the_prefix():
    W = wl.make("shared_prefix")
    sub = W.subset([2, 0])
    assert sub.prefix_len == W.prefix_len and sub.num_seqs == 2
    assert np.array_equal(sub.context_kv(0, 1)[0], W.context_kv(2, 1)[0])
    assert np.array_equal(sub.q_bits_seq(1), W.q_bits_seq(0))
    assert np.all(sub.page_table[:, :W.prefix_len // 16] == sub.page_table[0, :W.prefix_len // 16])
    W16 = wl.make("batch16_32k")
    assert np.array_equal(W16.subset([7]).outlier_channels, W16.outlier_channels)


def test_pool_rotation_covers_twice_the_l2():
    assert bench.pool_copies_for(10 ** 10) == 1
    for nbytes in (70 * 10 ** 6, 125 * 10 ** 6, 200 * 10 ** 6):
        n = bench.pool_copies_for(nbytes)
        assert n * nbytes >= 2 * bench.L2_BYTES and (n - 1) * nbytes < 2 * bench.L2_BYTES
