"""The N > 1 path of bench.py on the CPU. The path shards by sequence with no
exchange, so N GPUs run N independent replicas; what is shared is the host
side that times them. Two gloo ranks, one process each as torchrun launches
them, run the same pieces bench.py uses:
- the rank environment and a page-table seed per replica;
- barriers on both sides of a timed region;
- the step time as the maximum over ranks;
- the whole-job rate (every rank's rows over the slowest rank's time);
- the reference arm, which runs on rank 0 only: other ranks return at once and
  print nothing."""
import contextlib
import io
import json
import os
import socket
import time

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

ROWS_PER_RANK = 32


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class RefArgs:
    steps = 4
    warmup = 3


def worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, local = bench.rank_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        bench.barrier(dist)
        t0 = time.time()
        time.sleep(0.05 * (1 + 2 * r))   # ranks of unequal speed
        ms_local = 1.0 + 2.0 * r          # rank r's own step time: 1 ms, 3 ms
        bench.barrier(dist)
        wall = time.time() - t0           # after the closing barrier: at least the slowest rank's sleep
        ms = bench.max_over_ranks(dist, ms_local, torch.device("cpu"))
        rate = bench.whole_job_rate(ROWS_PER_RANK, w, ms)
        printed = io.StringIO()
        with contextlib.redirect_stdout(printed):
            ref = bench.run_reference(RefArgs) if r != 0 else None
        with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
            json.dump({"world": w, "rank": r, "local": local, "ms": ms, "rate": rate, "wall": wall,
                       "seed": bench.replica_seed(7, r), "ref": ref, "printed": printed.getvalue()}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_the_replicas_as_one_job(tmp_path):
    world = 2
    mp.start_processes(worker, args=(world, free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert (d["world"], d["rank"], d["local"]) == (world, r, r)
        assert d["ms"] == 3.0                                       # the slowest rank's time, on every rank
        assert d["rate"] == pytest.approx(world * ROWS_PER_RANK / 3e-3)
        assert d["wall"] >= 0.15 - 1e-3                             # the barrier waited for the slow rank
    assert res[0]["seed"] != res[1]["seed"]                          # each replica its own page table
    assert res[1]["ref"] is None and res[1]["printed"] == ""        # the oracle arm: rank 0 only


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(None, 2.5, torch.device("cpu")) == 2.5
    bench.barrier(None)
    assert bench.whole_job_rate(32, 1, 0.5) == pytest.approx(64000.0)
    assert bench.replica_seed(7, 0) == 7
