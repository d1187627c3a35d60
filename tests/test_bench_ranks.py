"""bench.py's whole-job figures with two gloo ranks on the CPU: work is summed
over the ranks (each draws its own batch, so their tokens and visible pairs
differ) and times are the slowest rank's; a single process passes its own
values through."""
import os
import socket
import tempfile

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

WORLD = 2


def _worker(rank, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        import bench
        sums, maxes = bench.rank_totals([1.5 * (rank + 1), 262144 + 27 * rank, 7], [3.0 + rank, 100.0 - rank])
        _, e2e = bench.rank_totals([], [2.0 + 5 * rank])
        if rank == 0:
            np.savez(os.path.join(out_dir, "r.npz"), sums=sums, maxes=maxes, e2e=e2e)
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_rank_totals_sum_work_and_take_slowest_time():
    with tempfile.TemporaryDirectory() as d:
        mp.spawn(_worker, args=(_free_port(), d), nprocs=WORLD, join=True)
        r = dict(np.load(os.path.join(d, "r.npz")))
    assert r["sums"].tolist() == [4.5, 2 * 262144 + 27, 14.0]
    assert r["maxes"].tolist() == [4.0, 100.0]
    assert r["e2e"].tolist() == [7.0]


def test_rank_totals_single_process_pass_through():
    import bench
    assert not dist.is_initialized()
    assert bench.rank_totals([1, 2.5], [3]) == ([1.0, 2.5], [3.0])
    assert bench.rank_totals([], [4]) == ([], [4.0])
