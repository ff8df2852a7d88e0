"""The benchmark's multi-rank bookkeeping on CPU (gloo, world size 2).

With N GPUs the benchmark runs N independent replicas of the layer (it shards
by tokens with no exchange); the only cross-rank steps are a barrier and the
max over ranks of the timed duration.  These run here with the gloo backend.
"""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        slow = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")
        tps = bench.tokens_per_second(4096, world, slow)
        q.put((rank, slow, tps))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_throughput_gloo_world2():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert [r[1] for r in res] == [15.0, 15.0]           # both ranks see the slowest
    assert res[0][2] == pytest.approx(2 * 4096 / 15e-3)   # all tokens / slowest time


def test_single_process_is_identity():
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.tokens_per_second(64, 1, 2.0) == pytest.approx(32000.0)


def test_algorithmic_work_closed_form():
    from workloads import SHAPES
    s = SHAPES["mixtral"]
    w = bench.algorithmic_work(s, [1024] * 8)
    assert w["kept"] == 8192 and w["touched"] == 8
    assert w["flops_gate_up"] == 2.0 * 8192 * 2 * 14336 * 4096
    assert w["flops_down"] == 2.0 * 8192 * 14336 * 4096
    assert w["weight_bytes"] == 8 * 3 * 4096 * 14336 * 2 + 8 * 4096 * 2
