"""The benchmark's multi-rank host logic on CPU with two gloo ranks: the
barrier, the max-over-ranks timing and the whole-job throughput. Heads are
independent, so ranks exchange nothing on the data path; only these timing
reductions cross ranks."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench._DIST["on"] = True
    bench.barrier()
    m = bench.max_over_ranks(10.0 * (rank + 1))
    v = bench.job_tflops(1e12, 4, m, bench.world())
    out[rank] = (bench.rank(), bench.world(), m, v)
    bench.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    assert sorted(out.keys()) == [0, 1]
    for r in range(world):
        rk, ws, m, v = out[r]
        assert rk == r and ws == world
        assert m == 20.0  # the slowest rank's time
        # 2 ranks x 4 steps x 1 TFLOP in 20 ms
        assert abs(v - 2 * 4 * 1.0 / 0.020) < 1e-9
