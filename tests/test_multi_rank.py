"""The bench's multi-rank path on the CPU: world-size-2 gloo process groups.

Under torchrun every rank times its own replica of the workload (the path shards into
independent replicas; no data-path collective). The whole-job figures are the slowest rank's
time and the units of all ranks, which is what `bench.reduce_over_ranks` returns on every
rank.
"""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir, ms, units):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        got = bench.reduce_over_ranks(ms[rank], units[rank], world, "cpu")
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{got[0]!r} {got[1]!r}\n")
    finally:
        dist.destroy_process_group()


def _run(tmp_path, ms, units):
    world = len(ms)
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path), ms, units),
                       nprocs=world, join=True, start_method="spawn")
    res = []
    for r in range(world):
        a, b = open(tmp_path / f"rank{r}.txt").read().split()
        res.append((float(a), float(b)))
    return res


def test_two_ranks_reduce_to_the_slowest_time_and_all_units(tmp_path):
    res = _run(tmp_path, ms=[812.5, 830.25], units=[4.0e12, 4.5e12])
    assert res == [(830.25, 8.5e12)] * 2  # every rank holds the whole-job figures


def test_the_slowest_rank_may_be_rank_zero(tmp_path):
    res = _run(tmp_path, ms=[9.0, 3.0], units=[1.0, 2.0])
    assert res == [(9.0, 3.0)] * 2


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(5.5, 7.0, 1, "cpu") == (5.5, 7.0)
