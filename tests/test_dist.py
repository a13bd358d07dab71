"""Replicas on several GPUs: the rank plumbing of bench.py on CPU (gloo, world size 2).

The decode path does not shard (one sequence per GPU, no collective on the data path); what runs
across ranks is the timing harness: process-group set-up, the barriers around the timed region,
the max over ranks of the elapsed time and the whole-job aggregate.  These tests run two processes
with the gloo backend on 127.0.0.1.
"""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str) -> None:
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_setup(None)
    elapsed_ms = 100.0 * (r + 1)  # rank 1 is the slower one
    bench.barrier(w)
    slowest = bench.max_over_ranks(elapsed_ms, w)
    value = bench.aggregate_tokens_per_s(w, steps=4, gen=256, ms_max=slowest)
    bench.barrier(w)
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "local": local, "backend": dist.get_backend(),
                   "slowest": slowest, "value": value}, f)
    dist.destroy_process_group()


def test_gloo_world2_barrier_max_and_aggregate(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, x in enumerate(res):
        assert (x["world"], x["rank"], x["local"], x["backend"]) == (2, r, r, "gloo")
        assert x["slowest"] == 200.0  # every rank sees the max over ranks
        # whole-job tokens/s: all ranks' tokens over the slowest rank's time
        assert x["value"] == pytest.approx(2 * 4 * 256 / 0.2)


def test_aggregate_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_tokens_per_s(1, steps=10, gen=256, ms_max=5000.0) == pytest.approx(512.0)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    """Under torchrun only rank 0 runs the (CPU) reference arm; the others return 0 at once."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = bench.argparse.Namespace(workload="tiny_f32_n2", alpha=None, steps=1, warmup=0, gpus=2)
    assert bench.main_reference(args) == 0
    assert capsys.readouterr().out == ""
