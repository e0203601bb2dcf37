"""The N > 1 host logic of the benchmark on CPU: world_size-2 gloo ranks agree
on the max time and on the weak-scaling whole-job throughput."""
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


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    ms = [10.0, 12.5][rank]
    mx = bench.barrier_max(ms, ws)
    val = bench.whole_job_tflops(1e12, 4, mx, ws)
    q.put((rank, mx, val))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, val in out:
        assert mx == 12.5
        assert val == pytest.approx(2 * 1e12 * 4 / 12.5e-3 / 1e12)
