"""The multi-rank side of bench.py on the CPU: two gloo ranks, each timing its
own instance of the workload; the job reports all ranks' work over the
slowest rank's time (weak scaling, no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch
    import torch.distributed as dist
    import bench
    from seeded_inputs import WORKLOADS
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    slowest = bench.max_over_ranks(ms, dist, torch.device("cpu"))
    w = WORKLOADS["sd21_unet_block"]
    out[rank] = (slowest, bench.whole_job_tflops(world, 1e12, 4, slowest), bench.rank_seed(w, rank))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    # 2 ranks x 4 steps x 1 TFLOP in 15 ms
    assert res[0][1] == pytest.approx(2 * 4 * 1.0 / 15e-3)
    assert res[0][2] != res[1][2]  # each rank draws its own instance


def test_single_process_is_unchanged():
    import bench
    assert bench.max_over_ranks(7.5, None, None) == 7.5


def test_percentile_and_cpu_model_helpers():
    import bench
    xs = [5.0, 1.0, 3.0, 2.0, 4.0]
    assert bench.percentile(xs, 0) == 1.0 and bench.percentile(xs, 100) == 5.0
    assert bench.percentile(xs, 50) == 3.0
    assert abs(bench.percentile(xs, 10) - 1.4) < 1e-12
    assert bench.percentile([7.0], 90) == 7.0 and bench.percentile([], 50) is None
    m = bench.host_cpu_model()
    assert isinstance(m, str) and m.endswith(")")
