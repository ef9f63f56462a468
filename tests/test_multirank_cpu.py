"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

Every rank runs an independent replica of the workload; the only
cross-rank steps are the barrier around the timed region and the max over
ranks of the measured time, which these tests exercise without a GPU.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        bench.barrier(ws)
        # rank-specific "times": the job time is the slowest rank's
        t = bench.reduce_max(10.0 + 5.0 * rank, ws, torch.device("cpu"))
        bench.barrier(ws)
        q.put((rank, t))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_ranks_barrier_and_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = dict(q.get(timeout=5) for _ in range(2))
    assert got == {0: 15.0, 1: 15.0}


def test_single_rank_helpers_are_identity():
    import bench
    assert bench.reduce_max(3.5, 1, torch.device("cpu")) == 3.5
    bench.barrier(1)
    w = bench.WORKLOADS["decode_ragged_b16_h32_n64k_d128_bf16"]
    lens = [3, 5] + [0] * 14
    assert bench.kv_bytes(w, lens) == 2 * 32 * 128 * 2 * 8
    assert bench.algorithmic_bytes(w, lens) > bench.kv_bytes(w, lens)
