"""The N > 1 path of bench.py on CPU: two gloo ranks stand in for two GPU
replicas.  Checks the max-over-ranks timing, the whole-job throughput, and
that only rank 0 runs the reference (oracle) arm."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [3.0, 5.5][rank]
    ms = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
    value = bench.job_tflops(world, bench.N_GEMMS * bench.GEMM_FLOPS, ms)

    class A:
        warmup, steps, cpu_budget = 0, 1, 0.1
    ref = bench.run_reference(A, rank, world) if rank == 1 else "skipped"
    out[rank] = (ms, value, ref)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 5.5
    expect = 2 * bench.N_GEMMS * bench.GEMM_FLOPS / 5.5e-3 / 1e12
    assert res[0][1] == pytest.approx(expect) and res[1][1] == pytest.approx(expect)
    assert res[1][2] is None  # the reference arm runs on rank 0 only


def test_single_rank_is_identity():
    assert bench.max_over_ranks(2.5, 1, None) == 2.5
    assert bench.job_tflops(1, 1e12, 1.0) == pytest.approx(1000.0)
