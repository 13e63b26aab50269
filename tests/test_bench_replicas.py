"""bench.py's N > 1 path on the CPU: two gloo ranks, as torchrun launches the
replicas.  Every rank runs the whole workload; the line reports the tokens of
all ranks over the slowest rank's time (no data-path collective)."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # rank r took (1 + r) s on the device and (10 - r) s end to end
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank], "cpu")
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(" ".join(repr(v) for v in got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    world = 2
    mp.spawn(_rank, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        vals = [float(v) for v in (tmp_path / f"rank{r}.txt").read_text().split()]
        assert vals == [2.0, 10.0]  # every rank sees the slowest replica's times


def test_max_over_ranks_without_a_group_is_the_identity():
    assert not dist.is_initialized()
    assert bench.max_over_ranks([3.5, 1.25], "cpu") == [3.5, 1.25]


def test_replica_tokens_count_every_rank():
    # llada8b_b1: batch 1, 1024 generated tokens; 2 replicas, 3 timed steps
    assert bench.replica_tokens(2, 3, 1, 1024) == 6144
    assert bench.replica_tokens(1, 3, 16, 256) == 12288
