"""bench.py's multi-rank host logic on CPU: world_size 2 over gloo.

Each rank is an independent replica (weak scaling, no data-path collective);
the only exchanges are the max-over-ranks of the step timings and the
agreement that every rank captured its CUDA graphs.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import sys
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench._dist()[:2] == (world, rank)
        # every rank owns a whole batch of its own (same shapes, its own seed)
        w = bench.rank_workload(rank)
        assert w.seed == rank and w.batch == 32 and w.fixed_len == 4096
        small = workloads.get("gqa_small", seed=rank)
        q = workloads.make_inputs(small).q
        qs = [torch.zeros_like(q) for _ in range(world)]
        dist.all_gather(qs, q)
        assert not torch.equal(qs[0], qs[1]), "replicas must not share inputs"
        # the only exchange: max over ranks of the per-rank timings
        mine = [1.0 + rank, 5.0 - rank, 2.0, 7.0 * (rank + 1)]
        got = bench.max_over_ranks(mine, torch.device("cpu"), world)
        assert got == [2.0, 5.0, 2.0, 14.0]
        # CUDA-graph timing: used only if every rank captured its graphs
        assert bench.all_ranks_ok(True, torch.device("cpu"), world)
        assert not bench.all_ranks_ok(rank == 0, torch.device("cpu"), world)
        vals, g = bench.merge_timings([1.0 + rank], 3.0 + rank, torch.device("cpu"), world)
        assert vals == [2.0] and g == 4.0
        vals, g = bench.merge_timings([1.0 + rank], None if rank == 1 else 3.0, torch.device("cpu"), world)
        assert vals == [2.0] and g is None
        # whole-job value: all ranks' bytes over the slowest step
        assert abs(bench.whole_job_gbs(world, 140_509_184, got[0]) - 2 * 140_509_184 / 2e-3 / 1e9) < 1e-9
    finally:
        dist.destroy_process_group()


def test_two_rank_weak_scaling_host_logic():
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port), nprocs=2, join=True, start_method="spawn")


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.0], torch.device("cpu"), 1) == [3.0, 4.0]
    assert bench.merge_timings([3.0], None, torch.device("cpu"), 1) == ([3.0], None)
    assert bench.merge_timings([3.0], 2.5, torch.device("cpu"), 1) == ([3.0], 2.5)
    assert bench.all_ranks_ok(True, torch.device("cpu"), 1) and not bench.all_ranks_ok(False, torch.device("cpu"), 1)
    assert bench.whole_job_gbs(1, 1_000_000_000, 1000.0) == pytest.approx(1.0)


def _bench(*args, timeout=300):
    import json
    import subprocess
    import sys
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    env["CUDA_VISIBLE_DEVICES"] = ""
    proc = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                          stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, timeout=timeout)
    lines = [json.loads(x) for x in proc.stdout.splitlines() if x.startswith("{")]
    return proc.returncode, lines, proc.stderr


def test_gpus_flag_self_launches_ranks():
    # no launcher: `bench.py --gpus 2` starts the two ranks itself; the dry run
    # takes the multi-rank host path (gloo) and rank 0 alone prints the line
    rc, lines, err = _bench("--gpus", "2", "--dry-run")
    assert rc == 0, err
    assert len(lines) == 1
    line = lines[0]
    assert line["dry_run"] and line["n_gpus"] == 2
    assert line["max_step_ms"] == 2.0      # max over ranks of 1 + rank
    assert line["max_seed"] == 1.0         # rank 1 drew its own replica


def test_gpus_flag_refuses_more_ranks_than_gpus():
    rc, lines, _ = _bench("--gpus", "2")
    assert rc == 2
    assert lines and "needs 2 visible GPUs" in lines[0]["error"]
