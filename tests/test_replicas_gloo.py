"""The N-GPU benchmark runs independent replicas (tokens are independent; no
collective on the data path).  Its host-side logic is checked here on CPU
with two gloo ranks: the barrier, the slowest-rank timing behind the
whole-job throughput, and the per-rank inputs (own batch, shared weights)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from mixture_experts_transformer_sigmoid_b300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
W = wl.Workload("replica", T=16, d=64, E=4, I=64, Is=64, k=2, routed_scale=1.0, dtype="bf16")


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _worker(rank, world, port, queue):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier(world)
        ms_max, value = bench.replica_throughput(world, W.T, 2.0 + rank)   # rank 1 is slower
        inp = bench.replica_inputs(W, rank, "cpu")
        queue.put((rank, ms_max, value, inp["x"].float().sum().item(),
                   inp["gate_up"].float().sum().item()))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_share_weights():
    world = 2
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, queue)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(queue.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ms0, v0, x0, g0), (r1, ms1, v1, x1, g1) = res
    assert ms0 == ms1 == pytest.approx(3.0)                  # the slowest rank's time
    assert v0 == v1 == pytest.approx(world * W.T / 3e-3)     # all ranks' tokens over it
    assert x0 != x1                                          # each replica its own batch
    assert g0 == g1                                          # the same weights
