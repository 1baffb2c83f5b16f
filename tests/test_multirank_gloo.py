"""The N-GPU bench path on the CPU: two gloo ranks.  Units shard across
ranks with no data exchange; the only cross-rank traffic is the barrier and
the max over ranks of the step time, and the whole-job value counts every
rank's batch."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workload as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 0.100 + 0.025 * rank          # rank 1 is the slower one
        local_e2e = 0.200 - 0.050 * rank         # rank 0 is slower end to end
        dist.barrier()
        max_ms, max_e2e = bench.slowest_rank(torch, local_ms, local_e2e, world, "cpu")
        none_ms, none_e2e = bench.slowest_rank(torch, local_ms, None, world, "cpu")
        q.put((rank, max_ms, max_e2e, none_ms, none_e2e))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, max_ms, max_e2e, none_ms, none_e2e in got:
        assert max_ms == pytest.approx(0.125)
        assert max_e2e == pytest.approx(0.200)
        assert none_ms == pytest.approx(0.125) and none_e2e is None


def test_whole_job_value_counts_every_rank():
    w = W.get_workload("batch")
    one = bench.whole_job_value(w, 1, 0.1)
    assert one == pytest.approx(w.units * w.k / 0.1e-3)
    assert bench.whole_job_value(w, 4, 0.1) == pytest.approx(4 * one)
    # weak scaling with a slower slowest rank lowers the job value
    assert bench.whole_job_value(w, 2, 0.2) == pytest.approx(one)


def test_bench_starts_its_own_ranks():
    """`python bench.py --gpus 2` without torchrun starts two ranks itself;
    each takes its own contiguous range of units (rank r: units
    [r*U, (r+1)*U) of the job), and rank 0 reports the job over both."""
    import json
    import subprocess
    import sys
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--gpus", "2",
                        "--_dry", "--workload", "tiny", "--steps", "3", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["n_gpus"] == 2
    w = W.get_workload("tiny")
    assert line["rank_units"] == [[0, w.units], [w.units, 2 * w.units]]
    assert line["value"] == pytest.approx(bench.whole_job_value(w, 2, line["ms_per_step"]))
