"""Replica (weak-scaling) host logic of the bench on CPU: two gloo ranks, each with its own
batch; the job throughput is the sum of tokens over the slowest rank's time. The path has no
data-path collective (units are independent), so this is the whole multi-GPU story."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from linear_attention_chunked_conv1d_gb300.inputs import WORKLOADS, make_inputs
    wl = WORKLOADS["gdn_t100_h4_d64_f32"]
    inp = make_inputs(wl, device="cpu", seed=rank)  # each replica draws its own batch
    tokens = sum(inp["lengths"])
    ms = 2.0 + rank  # rank 1 is the slower one
    value, ms_max, n = bench.aggregate(tokens, ms, dist)
    q.put((rank, value, ms_max, n, float(inp["x"].float().sum())))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_aggregate_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (_, v0, m0, n0, x0), (_, v1, m1, n1, x1) = res
    assert n0 == n1 == 2
    assert m0 == m1 == pytest.approx(3.0)           # max over ranks
    assert v0 == v1 == pytest.approx(200 / 3.0e-3)  # 100 tokens per rank / slowest time
    assert x0 != x1                                  # different batches per replica


def test_single_process_aggregate():
    import bench
    value, ms, n = bench.aggregate(1000, 2.0)
    assert (value, ms, n) == (pytest.approx(5e5), 2.0, 1)
