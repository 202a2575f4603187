"""bench.py's multi-rank path on CPU (gloo, world size 2): every rank runs its
own replica, the job's time is the slowest rank's, and the throughput counts
all ranks' tokens."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 2.0 if rank == 0 else 5.0
    slowest = bench.reduce_max(ms, "cpu")
    q.put((rank, slowest, bench.job_throughput(256, slowest, world)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in res:
        assert slowest == 5.0
        assert value == pytest.approx(2 * 256 / 5e-3)


def test_single_process_identity():
    import bench
    assert bench.reduce_max(3.5, "cpu") == 3.5
    assert bench.job_throughput(256, 1.0, 1) == pytest.approx(256000.0)


def test_clock_sampler_follows_visible_devices(monkeypatch):
    # the sampler must query the physical GPU the process runs on
    import bench
    monkeypatch.delenv("CUDA_VISIBLE_DEVICES", raising=False)
    assert bench.smi_device(0) == "0"
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "5")
    assert bench.smi_device(0) == "5"
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "3, 6")
    assert bench.smi_device(1) == "6"
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "GPU-1234abcd-0000-1111-2222-333344445555")
    assert bench.smi_device(0).startswith("GPU-1234abcd")
