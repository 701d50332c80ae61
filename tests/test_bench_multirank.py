"""The multi-rank host logic of bench.py on CPU: two gloo ranks, no GPU.

Under torchrun every rank runs its own, independently seeded batch (no
data-path collective); the job's time is the slowest rank's and its value
counts every rank's work.  The reference arm runs on rank 0 only."""
import argparse
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_path):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(10.0 * (rank + 1), "cpu")
    value = bench.job_value(world, 2e12, ms)
    # the reference arm: rank 0 alone does work and prints; the others return 0 at once
    args = argparse.Namespace(workload="tiny", steps=1, warmup=0, ref_budget=0.05)
    rc = bench.run_reference(args) if rank != 0 else 0
    dist.barrier()
    dist.destroy_process_group()
    with open(f"{out_path}.{rank}", "w") as f:
        f.write(f"{ms} {value} {rc}\n")


def test_two_gloo_ranks_take_the_slowest_time_and_count_all_work(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    out = str(tmp_path / "r")
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    for rank in range(2):
        ms, value, rc = open(f"{out}.{rank}").read().split()
        assert float(ms) == 20.0                      # max over ranks, identical on every rank
        assert abs(float(value) - 2 * 2e12 / 20e-3 / 1e12) < 1e-9
        assert int(rc) == 0


def test_single_rank_value_and_time_pass_through():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5, "cpu") == 7.5
    assert abs(bench.job_value(1, 43.6476051456e12, 64.5) - 676.7) < 0.1


def test_ranks_draw_independent_batches():
    from block_sparse_top_attn_gb300 import workloads as W
    a = W.make_problem("tiny", seed=0, values=False)
    b = W.make_problem("tiny", seed=1, values=False)
    assert a.sel.shape == b.sel.shape
    assert not np.array_equal(a.sel, b.sel)


def test_traffic_record_applies_only_to_its_workload_and_tiling(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    import json
    rec_path = tmp_path / "traffic.json"
    rec = {"source_sha1": bench.kernel_source_sha1(),
           "scaled": {"long128k/tile1024": {"bytes_per_launch": 2.5e10, "how": "test"}}}
    rec_path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_RECORD", str(rec_path))
    assert bench.traffic_record("long128k", 1024)[0] == 2.5e10
    assert bench.traffic_record("single8k", 0)[0] is None
    assert bench.traffic_record("long128k", 512)[0] is None
    rec["source_sha1"] = "0" * 40                      # counters of another build of the kernel
    rec_path.write_text(json.dumps(rec))
    value, why = bench.traffic_record("long128k", 1024)
    assert value is None and "changed" in why
    monkeypatch.setattr(bench, "TRAFFIC_RECORD", str(tmp_path / "missing.json"))
    assert bench.traffic_record("long128k", 1024)[0] is None
