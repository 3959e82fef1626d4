"""The multi-process path of bench.py on CPU: two ranks over gloo, each an
independent replica.  The job's time is the slowest rank's and its
throughput counts the units of every rank (no data-path collective; the path
does not shard)."""
import os
import sys

import pytest

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out_path):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 10.0 + 5.0 * rank                     # rank 1 is the slow one
    slow = bench.max_over_ranks(ms, world, device="cpu")
    value = bench.job_throughput(100, world, slow)  # 100 layer-steps per rank
    with open(f"{out_path}.{rank}", "w") as f:
        f.write(f"{slow} {value}\n")
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank(tmp_path):
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    out = str(tmp_path / "r")
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    for rank in range(2):
        slow, value = map(float, open(f"{out}.{rank}").read().split())
        assert slow == 15.0
        assert value == pytest.approx(2 * 100 / 15e-3)


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.job_throughput(10, 1, 5.0) == pytest.approx(2000.0)
