"""The multi-rank path of bench.py on CPU: two gloo ranks check the whole-job
aggregation (step time = max over ranks, work = sum over ranks) and that the
reference arm runs on rank 0 only."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, queue):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t_ms, tflops = bench.aggregate(local_ms=1.0 + rank, local_flops=1e12 * (rank + 1), steps=1,
                                   distributed=True)
    # the reference arm: rank 0 alone does work; others return 0 at once
    ref_rc = None
    if rank == 1:
        import argparse
        args = argparse.Namespace(steps=1, warmup=3, gpus=world)
        ref_rc = bench.run_reference(args, None, 0.05, 0.0)
    dist.barrier()
    dist.destroy_process_group()
    queue.put((rank, t_ms, tflops, ref_rc))


def test_two_rank_aggregation_gloo():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = {}
    for _ in procs:
        rank, t_ms, tflops, ref_rc = queue.get(timeout=120)
        results[rank] = (t_ms, tflops, ref_rc)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in (0, 1):
        t_ms, tflops, _ = results[rank]
        assert t_ms == pytest.approx(2.0)               # the slower rank's time
        assert tflops == pytest.approx(3e12 / 2e-3 / 1e12)  # all ranks' work / that time
    assert results[1][2] == 0
