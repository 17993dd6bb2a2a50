"""The benchmark's multi-rank helpers on CPU: two gloo ranks launched the way
torchrun launches them (RANK / WORLD_SIZE / MASTER_* in the environment).
Each rank holds an independent shard, so the only cross-rank steps are the
max of the timed spans and the sum of the rows; the reference arm runs on
rank 0 alone."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench

    class Args:
        pass

    w, r, local = bench.dist_setup(Args())
    assert (w, r, local) == (world, rank, rank)
    assert dist.get_backend() == "gloo"
    # rank r timed (r + 1) * 1.5 ms and owns 1000 * (r + 1) rows
    t = bench.max_over_ranks((rank + 1) * 1.5, world)
    n = bench.sum_over_ranks(1000.0 * (rank + 1), world)
    bench.barrier(world)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{t} {n}\n")
    dist.destroy_process_group()
    del torch


def test_two_gloo_ranks_max_time_and_summed_rows(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path)))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
            p.join()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    for r in range(world):
        t, n = map(float, (tmp_path / f"rank{r}.txt").read_text().split())
        assert t == pytest.approx(3.0)          # max over ranks of 1.5, 3.0
        assert n == pytest.approx(3000.0)       # 1000 + 2000 rows


def test_single_rank_helpers_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.sum_over_ranks(7.0, 1) == 7.0
