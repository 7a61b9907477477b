"""The N > 1 path of bench.py on CPU: two ranks over gloo, as torchrun would
start them (replicas only: no data-path collective).  The barrier and the
max-over-ranks timing work across ranks, every rank ends with the same
slowest time, the whole-job value counts every rank's bytes, and the
reference arm runs on rank 0 alone."""
import os
import socket
import sys
import types

import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    ws, r = bench.dist_setup()
    assert (ws, r) == (world, rank) and dist.get_backend() == "gloo"
    bench.barrier(ws)
    # each rank's own step time; all of them must see the slowest
    slowest = bench.max_over_ranks(1.0 + rank * 0.25, ws)
    value = bench.whole_job_gbs(2.0e9, slowest, ws)
    # the reference arm does nothing on ranks other than 0 (and returns)
    if rank != 0:
        assert bench.run_reference(types.SimpleNamespace(steps=1, warmup=0)) is None
    bench.barrier(ws)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{slowest} {value}\n")
    dist.destroy_process_group()


def test_two_gloo_ranks_share_the_slowest_time_and_sum_the_bytes(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    rows = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    slowest = 1.0 + (world - 1) * 0.25
    for s, v in rows:
        assert float(s) == slowest
        # 2 ranks x 2 GB per step over the slowest step time
        assert abs(float(v) - world * 2.0e9 / (slowest * 1e-3) / 1e9) < 1e-6
