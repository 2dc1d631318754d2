"""The N > 1 host path of bench.py on CPU: two gloo ranks (spawned processes).

Rows are independent, so each rank runs a replica of the workload and only
host-side coordination crosses ranks: a barrier around the timed region and
the maximum of the per-rank times, from which rank 0 reports the whole-job
throughput.  The reference arm runs on rank 0 only; other ranks exit without
work.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    # per-rank step times differ; every rank must see the slowest one
    t = bench.max_over_ranks(w, 1.0 + rank)
    # the reference arm returns at once on ranks other than 0 (it would
    # fail on the empty arguments if it did any work there)
    if rank != 0:
        bench.run_reference(object(), w, rank)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{w} {r} {t}\n")
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_share_max_time(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    for rank in range(world):
        w, r, t = open(tmp_path / f"rank{rank}.txt").read().split()
        assert int(w) == world and int(r) == rank
        assert float(t) == pytest.approx(2.0)          # max over ranks of 1.0, 2.0
