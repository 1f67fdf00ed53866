"""Replica scaling host logic with two gloo ranks on the CPU.

The decode path shards by requests with no collective: each rank decodes its
own batch of the same shape, and the benchmark reports the slowest rank's time
against all ranks' bytes. This checks the per-rank workloads and the
max-over-ranks reduction without a GPU.
"""

from __future__ import annotations

import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from workloads import config3_lengths, make_decode_workload
    w = make_decode_workload("r", config3_lengths(16), 32, 8, 128, 16, seed=100 + rank)
    got = bench.max_over_ranks(10.0 + rank)
    q.put((rank, got, int(w.q[0, 0, 0]), int(w.context_lens.sum())))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [11.0, 11.0]          # both ranks see the slowest
    assert res[0][3] == res[1][3]                        # same shape on every rank
    assert res[0][2] != res[1][2]                        # different values


def test_single_process_max_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
