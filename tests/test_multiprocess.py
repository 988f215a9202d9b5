"""The N > 1 host logic of bench.py on CPU: two gloo ranks.

The layer runs as independent replicas (no data-path collective); what the
bench does across ranks is a barrier and the whole-job aggregation: the sum of
the ranks' work over the slowest rank's time.  The reference arm runs on
rank 0 only.
"""

import io
import os
import socket
import contextlib
import types

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, local, w = bench.dist_info()
    assert (r, local, w) == (rank, rank, world)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    # rank r processed (r + 1) units in 10 (r + 1) ms
    units, ms = bench.aggregate(world, float(rank + 1), 10.0 * (rank + 1))
    bench.barrier(world)
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
        f.write(f"{units} {ms}\n")


def test_two_gloo_ranks_aggregate_sum_over_max(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    for r in range(world):
        units, ms = map(float, open(tmp_path / f"r{r}.txt").read().split())
        assert units == 3.0 and ms == 20.0


def test_single_rank_aggregate_is_identity():
    assert bench.aggregate(1, 5.0, 2.5) == (5.0, 2.5)


def test_reference_arm_runs_on_rank_zero_only():
    args = types.SimpleNamespace(steps=1, warmup=0)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, rank=1, local=1, world=2)
    assert buf.getvalue() == ""
