"""The benchmark's multi-process plumbing (replicas only: barrier + max over ranks) on CPU
with the gloo backend and two ranks. The path has no data-path collective; each rank runs
its own copy of the workload, and the job's time is the slowest rank's."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_init(backend="gloo")
    assert (r, w) == (rank, world)
    bench.barrier(w)
    slowest = bench.max_over_ranks(10.0 + rank, w, "cpu")
    bench.barrier(w)
    q.put((rank, slowest))
    dist.destroy_process_group()


def test_two_rank_barrier_and_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = dict(q.get(timeout=5) for _ in range(2))
    assert got == {0: 11.0, 1: 11.0}


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    bench.barrier(1)
    assert not dist.is_initialized() or torch.distributed.get_world_size() >= 1


def test_clock_summary_names_throttle_reasons():
    import bench
    # bits: 0x1 idle (not reported), 0x4 sw power cap, 0x40 hw thermal slowdown
    got = bench.ClockSampler.summarize([(2070.0, 0x0), (1980.0, 0x4), (2070.0, 0x41)], 2070.0)
    assert got["sm_mhz"] == 2070.0 and got["sm_max_mhz"] == 2070.0 and got["samples"] == 3
    assert got["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert bench.ClockSampler.summarize([], 2070.0) is None
